"""CPU oracle for the hand-written GPT-2 training step.  TEST INFRASTRUCTURE ONLY.

Only the test suite, the package entry's ``smoke()`` check and the benchmark's
CPU-baseline leg may import this module.  The CUDA library never calls it and
shares no code with it (the two see the same seeded inputs from
``step_gpt_train_03_b300.synth``, which draws random numbers and nothing else).

What it computes is the training step the llm.c pages describe:

* ujoy.net article, section "用C语言实现LLM" (implementing an LLM in C): one 1-D
  memory block allocated up front with every tensor pointing into it; a forward and
  a backward pass written by hand for each layer -- encoder, layernorm, matmul,
  self-attention, GELU, residual, softmax, cross-entropy -- chained together.
* same article, section "训练过程" (training run): forward, backward and an Adam
  update (lr 1e-4) chained into one loop; the printed model header
  (num_parameters 124439808, num_activations 73323776) fixes the architecture.
* yinghuohong.cn article, section "脚动完成每一个层前向/反向流传" (hand-written
  forward/backward of every layer): all memory allocated at the start, constant
  footprint, one flat array that weights and activations point into.

Readings where the pages are silent (each also listed in the design notes): GPT-2
pre-LN block with a final layernorm; LM head tied to the token table; linear
weights stored (out, in) with y = x W^T + b; layernorm eps 1e-5 inside the square
root with the biased variance; tanh-form GELU; attention scale 1/sqrt(hs) with a
causal mask; mean cross-entropy over all B*T positions computed over the V real
vocabulary columns (padded columns carry no probability and receive zero
gradient); AdamW with bias correction (t from 1), eps added after the square root,
decoupled weight decay applied to every parameter.

Every layer is a plain function on numpy arrays.  Matrix products use ``@`` (a
library routine); everything else is written out elementwise or as a plain
reduction, with no blocking or fusion.  The scalar type is a parameter: float64 by
default (parity), float32 to mirror the pages' fp32 program.
"""
from __future__ import annotations

import math

import numpy as np

PARAM_ORDER = (
    "wte", "wpe",
    "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
    "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb",
    "lnfw", "lnfb",
)

LN_EPS = 1e-5
GELU_SCALE = math.sqrt(2.0 / math.pi)


# --------------------------------------------------------------------------------------
# sizes: the pages' model header
# --------------------------------------------------------------------------------------
def param_shapes(max_seq_len, Vp, L, C):
    """Shape of every parameter tensor; the per-layer ones stacked over the L layers.

    ujoy.net article, section "训练过程": the header's num_parameters (124439808 at
    V=50257, C=768, L=12, maxT=1024) is met exactly by these sixteen tensors with an
    unpadded vocabulary, biases on every linear layer and no separate LM-head matrix.
    """
    return {
        "wte": (Vp, C), "wpe": (max_seq_len, C),
        "ln1w": (L, C), "ln1b": (L, C),
        "qkvw": (L, 3 * C, C), "qkvb": (L, 3 * C),
        "attprojw": (L, C, C), "attprojb": (L, C),
        "ln2w": (L, C), "ln2b": (L, C),
        "fcw": (L, 4 * C, C), "fcb": (L, 4 * C),
        "fcprojw": (L, C, 4 * C), "fcprojb": (L, C),
        "lnfw": (C,), "lnfb": (C,),
    }


def num_parameters(max_seq_len, V, L, C):
    """Element count of all parameter tensors (the pages' header prints this)."""
    return sum(int(np.prod(s)) for s in param_shapes(max_seq_len, V, L, C).values())


def activation_shapes(B, T, V, L, NH, C):
    """The activations the forward pass keeps, in the order the backward reads them.

    ujoy.net article, section "训练过程": num_activations 73323776 at B=4, T=64 is the
    element count of exactly this list (per-layer tensors stacked over L).
    """
    return {
        "encoded": (B, T, C),
        "ln1": (L, B, T, C), "ln1_mean": (L, B, T), "ln1_rstd": (L, B, T),
        "qkv": (L, B, T, 3 * C), "atty": (L, B, T, C),
        "preatt": (L, B, NH, T, T), "att": (L, B, NH, T, T),
        "attproj": (L, B, T, C), "residual2": (L, B, T, C),
        "ln2": (L, B, T, C), "ln2_mean": (L, B, T), "ln2_rstd": (L, B, T),
        "fch": (L, B, T, 4 * C), "fch_gelu": (L, B, T, 4 * C),
        "fcproj": (L, B, T, C), "residual3": (L, B, T, C),
        "lnf": (B, T, C), "lnf_mean": (B, T), "lnf_rstd": (B, T),
        "logits": (B, T, V), "probs": (B, T, V), "losses": (B, T),
    }


def num_activations(B, T, V, L, NH, C):
    return sum(int(np.prod(s)) for s in activation_shapes(B, T, V, L, NH, C).values())


# --------------------------------------------------------------------------------------
# layers (ujoy.net article, section "用C语言实现LLM": the layer list)
# --------------------------------------------------------------------------------------
def encoder_forward(tokens, wte, wpe):
    """Token plus position embedding: out[b,t,:] = wte[tokens[b,t],:] + wpe[t,:]."""
    B, T = tokens.shape
    return wte[tokens] + wpe[:T][None, :, :]


def encoder_backward(dwte, dwpe, dout, tokens):
    """Scatter-add of the output grad into the rows that were gathered (accumulates)."""
    B, T = tokens.shape
    for b in range(B):
        for t in range(T):
            dwte[tokens[b, t]] += dout[b, t]
    dwpe[:T] += dout.sum(axis=0)


def layernorm_forward(x, w, b):
    """Per row over the last axis: mean, biased variance, rstd = 1/sqrt(var + 1e-5);
    y = (x - mean) * rstd * w + b.  Returns (y, mean, rstd)."""
    mean = x.mean(axis=-1)
    xc = x - mean[..., None]
    var = (xc * xc).mean(axis=-1)
    rstd = 1.0 / np.sqrt(var + LN_EPS)
    xhat = xc * rstd[..., None]
    return xhat * w + b, mean, rstd


def layernorm_backward(dout, x, w, mean, rstd):
    """Grads of layernorm_forward.  With xhat = (x-mean)*rstd and g = dout*w:
    dx = rstd * (g - mean(g) - xhat * mean(g*xhat)); dw = sum dout*xhat; db = sum dout.
    Returns (dx, dw, db); dw and db are summed over every leading axis."""
    xhat = (x - mean[..., None]) * rstd[..., None]
    g = dout * w
    dx = rstd[..., None] * (g - g.mean(axis=-1, keepdims=True)
                            - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    C = x.shape[-1]
    dw = (dout * xhat).reshape(-1, C).sum(axis=0)
    db = dout.reshape(-1, C).sum(axis=0)
    return dx, dw, db


def matmul_forward(x, w, bias):
    """Linear layer with the weight stored (out, in): y = x @ w^T (+ bias)."""
    y = x @ w.T
    if bias is not None:
        y = y + bias
    return y


def matmul_backward(dout, x, w):
    """Grads of matmul_forward over the flattened rows: dx = dout @ w,
    dw = dout^T @ x, dbias = sum of dout over rows."""
    OC = dout.shape[-1]
    C = x.shape[-1]
    d2 = dout.reshape(-1, OC)
    x2 = x.reshape(-1, C)
    dx = (d2 @ w).reshape(x.shape)
    dw = d2.T @ x2
    db = d2.sum(axis=0)
    return dx, dw, db


def attention_forward(qkv, NH):
    """Causal multi-head self-attention.

    qkv[b,t] holds q, k, v as three C-wide thirds; head h uses columns
    [h*hs, (h+1)*hs) of each third.  preatt = q k^T / sqrt(hs) for key j <= query t
    (masked entries are -inf), att = row softmax of preatt, out = att v with the heads
    concatenated back to C columns.  Returns (out, preatt, att)."""
    B, T, C3 = qkv.shape
    C = C3 // 3
    hs = C // NH
    q = qkv[:, :, 0:C].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    k = qkv[:, :, C:2 * C].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    v = qkv[:, :, 2 * C:3 * C].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    scale = 1.0 / math.sqrt(hs)
    preatt = (q @ k.transpose(0, 1, 3, 2)) * scale
    future = np.triu(np.ones((T, T), dtype=bool), k=1)
    preatt[:, :, future] = -np.inf
    m = preatt.max(axis=-1, keepdims=True)
    e = np.exp(preatt - m)
    att = e / e.sum(axis=-1, keepdims=True)
    out = (att @ v).transpose(0, 2, 1, 3).reshape(B, T, C)
    return out, preatt, att


def attention_backward(dout, qkv, att, NH):
    """Grads of attention_forward with respect to qkv.

    dV = att^T dO; datt = dO V^T; softmax backward dS = att * (datt - rowsum(att*datt));
    dQ = dS K / sqrt(hs); dK = dS^T Q / sqrt(hs).  Masked entries have att = 0 and so
    get no gradient."""
    B, T, C3 = qkv.shape
    C = C3 // 3
    hs = C // NH
    q = qkv[:, :, 0:C].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    k = qkv[:, :, C:2 * C].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    v = qkv[:, :, 2 * C:3 * C].reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    do = dout.reshape(B, T, NH, hs).transpose(0, 2, 1, 3)
    scale = 1.0 / math.sqrt(hs)
    dv = att.transpose(0, 1, 3, 2) @ do
    datt = do @ v.transpose(0, 1, 3, 2)
    dpre = att * (datt - (att * datt).sum(axis=-1, keepdims=True))
    dq = (dpre @ k) * scale
    dk = (dpre.transpose(0, 1, 3, 2) @ q) * scale
    dqkv = np.empty_like(qkv)
    dqkv[:, :, 0:C] = dq.transpose(0, 2, 1, 3).reshape(B, T, C)
    dqkv[:, :, C:2 * C] = dk.transpose(0, 2, 1, 3).reshape(B, T, C)
    dqkv[:, :, 2 * C:3 * C] = dv.transpose(0, 2, 1, 3).reshape(B, T, C)
    return dqkv


def gelu_forward(x):
    """GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    u = GELU_SCALE * (x + 0.044715 * x * x * x)
    return 0.5 * x * (1.0 + np.tanh(u))


def gelu_backward(dout, x):
    """dx = dout * d/dx gelu(x), differentiating the tanh form term by term."""
    u = GELU_SCALE * (x + 0.044715 * x * x * x)
    th = np.tanh(u)
    sech2 = 1.0 - th * th
    du = GELU_SCALE * (1.0 + 3.0 * 0.044715 * x * x)
    return dout * (0.5 * (1.0 + th) + 0.5 * x * sech2 * du)


def residual_forward(a, b):
    return a + b


def softmax_forward(logits, V):
    """Probabilities over the first V (real) vocabulary columns; padded columns get 0."""
    z = logits[..., :V]
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    probs = np.zeros_like(logits)
    probs[..., :V] = e / e.sum(axis=-1, keepdims=True)
    return probs


def crossentropy_forward(probs, targets):
    """losses[b,t] = -log probs[b,t,targets[b,t]]."""
    B, T = targets.shape
    bi, ti = np.meshgrid(np.arange(B), np.arange(T), indexing="ij")
    return -np.log(probs[bi, ti, targets])


def crossentropy_softmax_backward(probs, targets, dloss):
    """d loss / d logits for loss = dloss-weighted sum of the per-position losses:
    dlogits = (probs - onehot(target)) * dloss[b,t]; padded columns stay 0."""
    B, T = targets.shape
    dlogits = probs * dloss[..., None]
    bi, ti = np.meshgrid(np.arange(B), np.arange(T), indexing="ij")
    dlogits[bi, ti, targets] -= dloss
    return dlogits


def adamw_update(params, grads, m, v, lr, beta1, beta2, eps, weight_decay, t):
    """One AdamW step over the flat buffer, in place.  ujoy.net article, section
    "训练过程": the demo fine-tunes with Adam at lr 1e-4 (weight_decay=0 is Adam).

    m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; mhat = m/(1-b1^t); vhat = v/(1-b2^t);
    p -= lr * (mhat / (sqrt(vhat) + eps) + wd * p)."""
    m *= beta1
    m += (1.0 - beta1) * grads
    v *= beta2
    v += (1.0 - beta2) * grads * grads
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    params -= lr * (mhat / (np.sqrt(vhat) + eps) + weight_decay * params)


# --------------------------------------------------------------------------------------
# the model: layers chained into forward / zero_grad / backward / update
# --------------------------------------------------------------------------------------
# ----------------------------------------------------------------- sampling and files
# The llm.c article, section "训练过程" (training run): after the fine-tuning loop the
# program generates samples from the model, and it starts from a checkpoint file of
# the weights written for the C program to load.  The pages give neither the sampler
# nor the file layout; the readings (inverse-CDF sampling driven by SplitMix64, and a
# 256-word int32 header followed by the fp32 tensors in parameter order) are in the
# design notes.

_M64 = (1 << 64) - 1


def splitmix64(seed, i):
    """Output i (i >= 1) of the SplitMix64 generator started at `seed`, from its published
    definition (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014): the state advances by the golden-ratio increment 0x9E3779B97F4A7C15 and
    the output is the state mixed by (z ^ z>>30) * 0xBF58476D1CE4E5B9,
    (z ^ z>>27) * 0x94D049BB133111EB, z ^ z>>31, all modulo 2^64."""
    z = (seed + i * 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def sample_token(z, V, temperature, seed, b):
    """Inverse-CDF draw from softmax(z[:V] / temperature) for sequence b: u = top 53 bits
    of SplitMix64 output b+1 over 2^53; the token is the first j whose running sum of
    exp((z_j - max) / temperature) exceeds u times the total.  Returns (token, lo, hi,
    threshold, total): [lo, hi) is the token's interval of the running sum."""
    x = np.asarray(z[:V], dtype=np.float64)
    e = np.exp((x - x.max()) / temperature)
    c = np.cumsum(e)
    u = (splitmix64(seed, b + 1) >> 11) / float(1 << 53)
    thr = u * c[-1]
    k = int(np.searchsorted(c, thr, side="right"))
    k = min(k, V - 1)
    lo = 0.0 if k == 0 else float(c[k - 1])
    return k, lo, float(c[k]), thr, float(c[-1])


# --------------------------------------------------------------------------------------
# fp8 (e4m3) quantization: the lower-precision variant (yinghuohong.cn article, section
# "脚动完成每一个层前向/反向流传": precision planned to go from fp32 down to fp16 or lower)
# --------------------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_value(code):
    """The real number an e4m3 byte stands for, from the format's definition: sign bit,
    4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
    (m/8 * 2^-6); S.1111.111 is NaN and there is no infinity, so the largest finite
    magnitude is 1.75 * 2^8 = 448."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)])


def e4m3_round(x):
    """Round to the nearest e4m3 value, ties to the even mantissa, saturating at +-448
    (finite inputs).  With e = floor(log2|x|) clamped to >= -6 (the subnormal range
    shares the spacing of the smallest binade), the grid spacing is 2^(e-3)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # log2 of values just below a power of two can land on it: correct by comparison
    e = np.where(2.0 ** e > a, e - 1, e)
    e = np.where(2.0 ** (e + 1) <= a, e + 1, e)
    e = np.maximum(e, -6.0)
    step = 2.0 ** (e - 3)
    r = np.round(a / step) * step            # numpy rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.sign(x) * r


def e4m3_encode(x):
    """Codes (uint8) of e4m3_round(x): the sign bit of x (a negative value that rounds to
    zero is -0) plus the index of the magnitude in the table of non-negative values
    (which is increasing)."""
    x = np.asarray(x, dtype=np.float64)
    r = e4m3_round(x)
    pos = E4M3_TABLE[:127]                    # codes 0x00..0x7E: 0 .. 448, increasing
    idx = np.searchsorted(pos, np.abs(r))
    return (idx | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def pow2_scale_exponent(amax):
    """The largest k with amax * 2^k <= 448 (amax > 0 finite; 0 for amax == 0): a
    power-of-two scale, so scaling and unscaling are exact.  With amax = f 2^e, f in
    [0.5, 1): k = 9 - e if f <= 0.875 (448 = 0.875 2^9), else 8 - e; clamped to
    [-126, 126] so that 2^k and 2^-k are normal fp32 numbers."""
    a = float(amax)
    if a == 0.0:
        return 0
    f, e = math.frexp(a)
    k = (9 - e) if f <= 0.875 else (8 - e)
    return max(-126, min(126, k))


def quantize_rows_e4m3(y):
    """Row-wise scaling: for each row, k = pow2_scale_exponent(max |y|), values
    e4m3_round(y * 2^k).  Returns (dequantized rows, codes, exponents k)."""
    y = np.asarray(y)
    rows = y.reshape(-1, y.shape[-1])
    ks = np.array([pow2_scale_exponent(np.abs(r).max()) for r in rows])
    scaled = rows * np.exp2(ks)[:, None]
    q = e4m3_round(scaled)
    deq = q * np.exp2(-ks)[:, None]
    return deq.reshape(y.shape), e4m3_encode(scaled).reshape(y.shape), ks


def quantize_tensor_e4m3(w):
    """Tensor-wise scaling: k = pow2_scale_exponent(max |w|), values e4m3_round(w 2^k).
    Returns (dequantized tensor, codes, k)."""
    w = np.asarray(w)
    k = pow2_scale_exponent(np.abs(w).max())
    scaled = w * 2.0 ** k
    return e4m3_round(scaled) * 2.0 ** -k, e4m3_encode(scaled), k


def matmul_forward_fp8(x, w, bias):
    """The fp8 linear layer: the input quantized row by row and the weight as one tensor
    (power-of-two scales, e4m3 values), multiplied exactly, then unscaled; the bias is
    added unquantized.  The backward of the layer is matmul_backward on the unquantized
    input and weight (the quantization passes gradients straight through)."""
    xq, _, _ = quantize_rows_e4m3(x)
    wq, _, _ = quantize_tensor_e4m3(w)
    return matmul_forward(xq, wq, bias)


# --------------------------------------------------------------------------------------
# Muon (pimou.com article, sections "优化器的优势" and "相关技术的追溯": the Muon optimizer
# orthogonalizes with Newton-Schulz iterations after Bernstein & Newhouse (2024))
# --------------------------------------------------------------------------------------
MUON_TENSORS = ("qkvw", "attprojw", "fcw", "fcprojw")   # the 2-D matrices of every block


def round_bf16(x):
    """Round to the nearest bfloat16 (ties to even), from the format's definition: the
    top 16 bits of the float32 encoding, the dropped 16 bits rounded to nearest even.
    Computed on the float32 value of x (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = (b >> 16) & 1
    b = (b + 0x7FFF + keep) >> 16 << 16
    return (b & 0xFFFFFFFF).astype(np.uint32).view(np.float32).astype(np.float64)


def newton_schulz(G, iters, bf16=False):
    """The cubic Newton-Schulz iteration towards the orthogonal polar factor of G: start
    from X = G / ||G||_F (all singular values in (0, 1]), then `iters` times
    X <- 1.5 X - 0.5 X X^T X, which maps each singular value s to 1.5 s - 0.5 s^3 and so
    drives every nonzero one towards 1 while keeping the singular vectors.  Written on
    the smaller Gram matrix: with S = X^T X (tall or square X) or X X^T (wide) and
    T = 1.5 I - 0.5 S, X <- X T or T X (the same product).

    bf16=True: the arithmetic of a bf16 implementation -- X, S and T rounded to bf16 where
    it stores them (X after the normalization and after every step), the products and
    sums exact.  Small singular values grow by 1.5 per step and so does the rounding in
    their directions, so the bf16 iterate drifts from the exact one as steps are added."""
    rnd = round_bf16 if bf16 else (lambda a: a)
    X = np.asarray(G, dtype=np.float64)
    nrm = np.sqrt((X * X).sum())
    if nrm == 0.0:
        return X.copy()
    X = rnd(X / nrm)
    tall = X.shape[0] >= X.shape[1]
    n = X.shape[1] if tall else X.shape[0]
    for _ in range(iters):
        S = rnd(X.T @ X if tall else X @ X.T)
        T = rnd(1.5 * np.eye(n) - 0.5 * S)
        X = rnd(X @ T if tall else T @ X)
    return X


def muon_update(params, grads, mom, lr, momentum, weight_decay, iters):
    """One Muon step on each matrix of MUON_TENSORS (per layer): mom <- momentum mom + g,
    O = newton_schulz(mom), p <- p - lr (O + weight_decay p)."""
    for name in MUON_TENSORS:
        for l in range(params[name].shape[0]):
            mom[name][l] = momentum * mom[name][l] + grads[name][l]
            O = newton_schulz(mom[name][l], iters)
            params[name][l] -= lr * (O + weight_decay * params[name][l])


PARAM_FILE_MAGIC = 20240326
PARAM_FILE_VERSION = 3


def read_param_file(path):
    """(header ints, {name: fp32 array} in parameter order) of a parameter file: 256
    little-endian int32 header words, then the tensors back to back.  The tensor
    shapes follow from the header's max_seq_len, padded vocab, layers and channels."""
    with open(path, "rb") as f:
        h = np.frombuffer(f.read(1024), dtype="<i4")
        rest = np.frombuffer(f.read(), dtype="<f4")
    max_seq_len, L, C, Vp = int(h[2]), int(h[4]), int(h[6]), int(h[7])
    out, off = {}, 0
    for name, shp in param_shapes(max_seq_len, Vp, L, C).items():
        n = int(np.prod(shp))
        out[name] = rest[off:off + n].reshape(shp)
        off += n
    if off != rest.size:
        raise ValueError(f"{rest.size - off} trailing values in {path}")
    return h, out


class GPT2Oracle:
    """GPT-2 over one flat parameter buffer (views carve it into tensors).

    yinghuohong.cn article, section "脚动完成每一个层前向/反向流传", and ujoy.net
    article, section "用C语言实现LLM": one 1-D block holds every weight, layers are
    chained into forward, backward and update.
    """

    def __init__(self, max_seq_len, V, Vp, L, NH, C, dtype=np.float64):
        self.maxT, self.V, self.Vp, self.L, self.NH, self.C = max_seq_len, V, Vp, L, NH, C
        self.dtype = np.dtype(dtype)
        self.shapes = param_shapes(max_seq_len, Vp, L, C)
        self.sizes = {k: int(np.prod(s)) for k, s in self.shapes.items()}
        self.num_params = sum(self.sizes.values())
        self.flat = np.zeros(self.num_params, self.dtype)
        self.flat_grad = np.zeros(self.num_params, self.dtype)
        self.m = np.zeros(self.num_params, self.dtype)
        self.v = np.zeros(self.num_params, self.dtype)
        self.p = self._views(self.flat)
        self.g = self._views(self.flat_grad)
        self.acts = None
        self.batch = None
        # the pre-softmax scores are part of the pages' activation list but the backward
        # does not read them; large runs may drop them to save host memory
        self.keep_preatt = True
        # fp8 variant: the two products whose input is a layernorm output (qkv, fc) take
        # e4m3 operands (matmul_forward_fp8); everything else as in the plain model
        self.fp8 = False

    def _views(self, flat):
        out, off = {}, 0
        for name in PARAM_ORDER:
            n = self.sizes[name]
            out[name] = flat[off:off + n].reshape(self.shapes[name])
            off += n
        return out

    def load(self, params: dict):
        for name in PARAM_ORDER:
            a = np.asarray(params[name])
            if a.shape != self.shapes[name]:
                raise ValueError(f"{name}: shape {a.shape} != {self.shapes[name]}")
            self.p[name][...] = a

    def forward(self, tokens, targets=None):
        """Forward pass; returns the mean loss (or None without targets)."""
        p, L, NH = self.p, self.L, self.NH
        tokens = np.asarray(tokens)
        B, T = tokens.shape
        if T > self.maxT:
            raise ValueError("T exceeds max_seq_len")
        if tokens.min() < 0 or tokens.max() >= self.V:
            raise ValueError("token id out of range")
        a = {"ln1": [], "ln1_mean": [], "ln1_rstd": [], "qkv": [], "atty": [], "preatt": [],
             "att": [], "attproj": [], "residual2": [], "ln2": [], "ln2_mean": [],
             "ln2_rstd": [], "fch": [], "fch_gelu": [], "fcproj": [], "residual3": []}
        x = encoder_forward(tokens, p["wte"], p["wpe"])
        a["encoded"] = x
        for l in range(L):
            ln1, m1, r1 = layernorm_forward(x, p["ln1w"][l], p["ln1b"][l])
            mm_in = matmul_forward_fp8 if self.fp8 else matmul_forward
            qkv = mm_in(ln1, p["qkvw"][l], p["qkvb"][l])
            atty, preatt, att = attention_forward(qkv, NH)
            attproj = matmul_forward(atty, p["attprojw"][l], p["attprojb"][l])
            res2 = residual_forward(x, attproj)
            ln2, m2, r2 = layernorm_forward(res2, p["ln2w"][l], p["ln2b"][l])
            fch = mm_in(ln2, p["fcw"][l], p["fcb"][l])
            g = gelu_forward(fch)
            fcproj = matmul_forward(g, p["fcprojw"][l], p["fcprojb"][l])
            res3 = residual_forward(res2, fcproj)
            if not self.keep_preatt:
                preatt = None
            for k_, v_ in (("ln1", ln1), ("ln1_mean", m1), ("ln1_rstd", r1), ("qkv", qkv),
                           ("atty", atty), ("preatt", preatt), ("att", att),
                           ("attproj", attproj), ("residual2", res2), ("ln2", ln2),
                           ("ln2_mean", m2), ("ln2_rstd", r2), ("fch", fch), ("fch_gelu", g),
                           ("fcproj", fcproj), ("residual3", res3)):
                a[k_].append(v_)
            x = res3
        lnf, mf, rf = layernorm_forward(x, p["lnfw"], p["lnfb"])
        a["lnf"], a["lnf_mean"], a["lnf_rstd"] = lnf, mf, rf
        logits = matmul_forward(lnf, p["wte"], None)     # tied LM head, no bias
        a["logits"] = logits
        self.acts = a
        self.batch = (tokens, None if targets is None else np.asarray(targets))
        if targets is None:
            a["probs"] = None
            return None
        probs = softmax_forward(logits, self.V)
        losses = crossentropy_forward(probs, np.asarray(targets))
        a["probs"], a["losses"] = probs, losses
        return float(losses.mean())

    def zero_grad(self):
        self.flat_grad[...] = 0.0

    def backward(self):
        """Backward of every layer in reverse; accumulates into the grad buffer."""
        if self.acts is None or self.batch[1] is None:
            raise RuntimeError("backward needs a forward pass with targets")
        a, p, g, L, NH = self.acts, self.p, self.g, self.L, self.NH
        tokens, targets = self.batch
        B, T = tokens.shape
        dloss = np.full((B, T), 1.0 / (B * T), dtype=self.dtype)   # d(mean)/d(loss_bt)
        dlogits = crossentropy_softmax_backward(a["probs"], targets, dloss)
        dlnf, dwte, _ = matmul_backward(dlogits, a["lnf"], p["wte"])
        g["wte"] += dwte
        x_last = a["residual3"][L - 1]
        dx, dw, db = layernorm_backward(dlnf, x_last, p["lnfw"], a["lnf_mean"], a["lnf_rstd"])
        g["lnfw"] += dw
        g["lnfb"] += db
        for l in reversed(range(L)):
            x_in = a["encoded"] if l == 0 else a["residual3"][l - 1]
            dres3 = dx
            # MLP branch: res3 = res2 + fcproj(gelu(fc(ln2(res2))))
            dg, dw, db = matmul_backward(dres3, a["fch_gelu"][l], p["fcprojw"][l])
            g["fcprojw"][l] += dw
            g["fcprojb"][l] += db
            dfch = gelu_backward(dg, a["fch"][l])
            dln2, dw, db = matmul_backward(dfch, a["ln2"][l], p["fcw"][l])
            g["fcw"][l] += dw
            g["fcb"][l] += db
            dres2_ln, dw, db = layernorm_backward(dln2, a["residual2"][l], p["ln2w"][l],
                                                  a["ln2_mean"][l], a["ln2_rstd"][l])
            g["ln2w"][l] += dw
            g["ln2b"][l] += db
            dres2 = dres3 + dres2_ln                       # residual: grad flows to both
            # attention branch: res2 = x + attproj(attn(qkv(ln1(x))))
            datty, dw, db = matmul_backward(dres2, a["atty"][l], p["attprojw"][l])
            g["attprojw"][l] += dw
            g["attprojb"][l] += db
            dqkv = attention_backward(datty, a["qkv"][l], a["att"][l], NH)
            dln1, dw, db = matmul_backward(dqkv, a["ln1"][l], p["qkvw"][l])
            g["qkvw"][l] += dw
            g["qkvb"][l] += db
            dx_ln, dw, db = layernorm_backward(dln1, x_in, p["ln1w"][l],
                                               a["ln1_mean"][l], a["ln1_rstd"][l])
            g["ln1w"][l] += dw
            g["ln1b"][l] += db
            dx = dres2 + dx_ln
        encoder_backward(g["wte"], g["wpe"], dx, tokens)

    def update(self, lr, beta1, beta2, eps, weight_decay, t):
        adamw_update(self.flat, self.flat_grad, self.m, self.v, lr, beta1, beta2, eps,
                     weight_decay, t)

    def update_muon(self, lr_muon, momentum, iters, lr, beta1, beta2, eps, weight_decay, t):
        """Muon on the block matrices (momentum kept in the AdamW first-moment buffer of
        those parameters), AdamW with (lr, beta1, beta2, eps, weight_decay) on every other
        parameter; weight_decay also applies, decoupled, in the Muon step."""
        other = np.ones(self.num_params, dtype=bool)
        off = 0
        for name in PARAM_ORDER:
            n = self.sizes[name]
            if name in MUON_TENSORS:
                other[off:off + n] = False
            off += n
        idx = np.nonzero(other)[0]
        p, g, m, v = self.flat[idx], self.flat_grad[idx], self.m[idx], self.v[idx]
        adamw_update(p, g, m, v, lr, beta1, beta2, eps, weight_decay, t)
        self.flat[idx], self.m[idx], self.v[idx] = p, m, v
        muon_update(self.p, self.g, self._views(self.m), lr_muon, momentum, weight_decay, iters)

    def step(self, tokens, targets, lr, beta1, beta2, eps, weight_decay, t):
        loss = self.forward(tokens, targets)
        self.zero_grad()
        self.backward()
        self.update(lr, beta1, beta2, eps, weight_decay, t)
        return loss

    def grads(self) -> dict:
        return self.g

    def params(self) -> dict:
        return self.p


def from_shape(shape, dtype=np.float64) -> GPT2Oracle:
    """Oracle for a ``synth.ModelShape``-like object (attribute access only)."""
    return GPT2Oracle(shape.max_seq_len, shape.vocab_size, shape.padded_vocab_size,
                      shape.num_layers, shape.num_heads, shape.channels, dtype)
