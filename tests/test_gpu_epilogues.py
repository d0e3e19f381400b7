"""Element-wise parity of the fused matmul epilogues and the weight-gradient reduction
paths of the tensor-core kernels, through the C ABI, against the CPU oracle (fp64).

The model's linear layers run as one kernel each with the next layer's elementwise work
fused into the epilogue (ujoy.net llm.c article, section "用C语言实现LLM": the matmul,
GELU and residual layers and their backward passes): bias, GELU (the pre-activation is
kept), the residual add, the GELU backward fused into the input gradient, fp32 weight
gradients added in place with a split contraction when a weight has few tiles.  Each is
compared here with the oracle's separate layers, at the 124M model's full sizes (16384
rows) -- every element, except for the LM head's 16384 x 50304 products, checked on
sampled rows that touch every output tile -- and on small ragged shapes.

Tolerances (max |got - ref| / max |ref|), from the arithmetic:
* bf16 outputs: the stored result is rounded to bf16 (relative error <= 2^-9 = 1.95e-3);
  products of bf16 inputs are exact in fp32 and accumulate in fp32 (relative ~1e-5 at
  K = 3072).  Bound 4e-3.
* GELU output: gelu of the stored (bf16) pre-activation h, so against the oracle's exact
  gelu(h) it carries the rounding of h (|gelu'| <= 1.13 times 2^-9 |h|), the rounding of
  the result (2^-9) and the hardware tanh (relative error 2^-11, at most 0.5 |h| 2^-11):
  (1.13 + 1 + 0.25) 2^-9 = 4.7e-3 where |gelu(h)| ~ |h| is largest.  Bound 6e-3.
* GELU backward: gelu'(x) = 0.5 (1 + th) + 0.5 x (1 - th^2) sqrt(2/pi) (1 + 3 0.044715 x^2)
  depends on th with slope up to ~10 for |x| <= 4, so the 2^-11 tanh error can move
  gelu' by up to ~5e-3; with the bf16 rounding of the result the bound is 1e-2.
* fp32 weight gradients: fp32 accumulation over up to 16384 rows, split contractions
  added in a fixed order: 1e-4 (as the other fp32 gradient checks).
* bias gradient summed in the GELU backward's output stage: against the exact (fp64)
  column sums of the stored dinp it differs only by fp32 summation, relative ~1e-7:
  bound 1e-5; against the oracle it carries dinp's errors, which average out over the
  rows: bound GELU_BWD_TOL.
"""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from tests.gpu_helpers import ensure_built, norm_err

pytestmark = pytest.mark.gpu

BF16_TOL = 4e-3
GELU_TOL = 6e-3
GELU_BWD_TOL = 1e-2
F32_TOL = 1e-4
FP32_OUT_TOL = 1e-5


@pytest.fixture(scope="module")
def G():
    ensure_built()
    import torch
    from step_gpt_train_03_b300 import gpt2lib
    torch.cuda.init()
    return gpt2lib


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _inputs(M, N, K, prec, seed, wscale=None):
    """x (M,K) ~ N(0,1), W (N,K) ~ N(0, wscale^2) with wscale = 1/sqrt(K) (pre-activations of
    unit scale, so GELU is exercised over its whole curve), bias ~ N(0, 0.1^2), residual
    (M,N) ~ N(0,1), on the GPU in the path's type; the oracle gets exactly those values."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    dt = torch.bfloat16 if prec == "bf16" else torch.float32
    ws = wscale if wscale is not None else 1.0 / np.sqrt(K)
    x = torch.randn(M, K, device="cuda", generator=g).to(dt)
    w = (ws * torch.randn(N, K, device="cuda", generator=g)).to(dt)
    b = (0.1 * torch.randn(N, device="cuda", generator=g)).to(dt)
    r = torch.randn(M, N, device="cuda", generator=g).to(dt)
    return x, w, b, r


def _samples(n, k, rng):
    """k indices in [0, n) spread over every 128-block, plus the last index."""
    idx = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    idx.update(range(0, n, 128))
    idx.add(n - 1)
    return np.array(sorted(idx))


# ------------------------------------------------------------------ full-size forward epilogues
@pytest.mark.parametrize("M,N,K,epi", [
    (16384, 3072, 768, "gelu"),        # fc: CTA pairs, GELU epilogue (pre-activation kept)
    (16384, 768, 3072, "residual"),    # MLP projection: CTA pairs, residual epilogue
    (16384, 768, 768, "residual"),     # attention projection: single CTAs, residual epilogue
    (16384, 2304, 768, "bias"),        # qkv: CTA pairs, bias only
])
def test_forward_epilogue_full_size(G, M, N, K, epi):
    """Every element of the output (and of the kept pre-activation) against the oracle's
    separate matmul, GELU and residual layers."""
    import torch
    x, w, b, r = _inputs(M, N, K, "bf16", seed=M + N + K)
    out = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    aux = torch.empty(M, N, device="cuda", dtype=torch.bfloat16) if epi == "gelu" else (r if epi == "residual" else None)
    G.matmul_forward_fused(out, aux, x, w, b, epi, "bf16")
    G.layer_check()
    h = O.matmul_forward(_f64(x), _f64(w), _f64(b))
    got = _f64(out)
    if epi == "bias":
        e = norm_err(got, h)
        assert e <= BF16_TOL, e
    elif epi == "residual":
        e = norm_err(got, O.residual_forward(_f64(r), h))
        assert e <= BF16_TOL, e
    else:
        e = norm_err(_f64(aux), h)
        assert e <= BF16_TOL, ("pre-activation", e)
        e = norm_err(got, O.gelu_forward(h))
        assert e <= GELU_TOL, ("gelu", e)
        # the pre-activations span the curve (not only its linear part)
        assert h.min() < -3 and h.max() > 3


def test_gelu_backward_input_gradient_full_size(G):
    """MLP projection backward: dh (16384, 3072) = (dres (16384, 768) Wfcproj (768, 3072))
    * gelu'(h), CTA pairs with the pre-activation read ahead by TMA."""
    import torch
    M, N, K = 16384, 768, 3072
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    dout = torch.randn(M, N, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) / np.sqrt(N)).to(torch.bfloat16)
    pre = (1.5 * torch.randn(M, K, device="cuda", generator=g)).to(torch.bfloat16)
    dinp = torch.empty(M, K, device="cuda", dtype=torch.bfloat16)
    db0 = torch.randn(K, device="cuda", generator=g)
    dbias = db0.clone()
    sc = torch.empty(G.matmul_backward_input_gelu_scratch_bytes(M, K), dtype=torch.uint8, device="cuda")
    G.matmul_backward_input_gelu(dinp, dout, w, pre, "bf16", dbias, sc)
    G.layer_check()
    ref = O.gelu_backward(_f64(dout) @ _f64(w), _f64(pre))
    got = _f64(dinp)
    e = norm_err(got, ref)
    assert e <= GELU_BWD_TOL, e
    # the fused bias gradient (added into dbias): the stored rows' column sums
    db = (dbias - db0).double().cpu().numpy()
    assert norm_err(db, got.sum(axis=0)) <= FP32_OUT_TOL
    assert norm_err(db, ref.sum(axis=0)) <= GELU_BWD_TOL


# ------------------------------------------------------------------ full-size weight gradients
@pytest.mark.parametrize("M,N,K", [
    (16384, 768, 768),       # attention projection: 9 pair tiles, contraction split 8 ways
    (16384, 3072, 768),      # fc: 36 pair tiles, split 2 ways
    (16384, 768, 3072),      # MLP projection
    (16384, 2304, 768),      # qkv
    (16384, 50304, 768),     # LM head (tied): 50304 x 768 weight gradient, 50304-wide dX contraction
])
def test_matmul_backward_full_size_sampled(G, M, N, K):
    """dX (bf16) and dW (fp32, added into existing values) and dbias of the model's
    linear layers at 16384 rows; dW of the few-tile weights takes the split contraction
    whose partial tiles are added in a fixed order."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(N + K)
    dout = torch.randn(M, N, device="cuda", generator=g).to(torch.bfloat16)
    x = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) / np.sqrt(N)).to(torch.bfloat16)
    dinp = torch.empty(M, K, device="cuda", dtype=torch.bfloat16)
    dW0 = torch.randn(N, K, device="cuda", generator=g)
    dW = dW0.clone()
    dB = torch.zeros(N, device="cuda")
    sc = torch.empty(G.matmul_backward_scratch_bytes(M, N), dtype=torch.uint8, device="cuda")
    G.matmul_backward(dinp, dW, dB, dout, x, w, "bf16", sc)
    G.layer_check()
    x64, w64 = _f64(x), _f64(w)
    rng = np.random.default_rng(K)
    rows, kcols, nrows = _samples(M, 32, rng), _samples(K, 32, rng), _samples(N, 32, rng)
    # the sampled rows of dX and of dW touch every output tile; for the widest products
    # (the LM head) the oracle reads only those slices of dout, not the whole 16384 x 50304
    d_rows = _f64(dout[torch.as_tensor(rows, device="cuda")])
    d_ncols = _f64(dout[:, torch.as_tensor(nrows, device="cuda")])
    got_dx = _f64(dinp)
    got_dw = (dW - dW0).double().cpu().numpy()
    assert norm_err(got_dx[rows], d_rows @ w64) <= BF16_TOL, "dX rows"
    assert norm_err(got_dw[nrows], d_ncols.T @ x64) <= F32_TOL, "dW rows"
    if N <= 4096:
        d64 = _f64(dout)
        assert norm_err(got_dx[:, kcols], d64 @ w64[:, kcols]) <= BF16_TOL, "dX columns"
        assert norm_err(got_dw[:, kcols], d64.T @ x64[:, kcols]) <= F32_TOL, "dW columns"
    db_ref = np.zeros(N)
    for i in range(0, M, 1024):
        db_ref += _f64(dout[i:i + 1024]).sum(axis=0)
    assert norm_err(dB.double().cpu().numpy(), db_ref) <= F32_TOL


# ------------------------------------------------------------------ ragged shapes, every element
@pytest.mark.parametrize("prec", ["bf16", "fp32"])
@pytest.mark.parametrize("M,N,K", [(300, 200, 136), (129, 264, 776), (1, 64, 64), (513, 1032, 520)])
def test_fused_epilogues_ragged_every_element(G, prec, M, N, K):
    import torch
    x, w, b, r = _inputs(M, N, K, prec, seed=7 * M + N)
    dt = x.dtype
    x64, w64, b64, r64 = _f64(x), _f64(w), _f64(b), _f64(r)
    h = O.matmul_forward(x64, w64, b64)
    tol = BF16_TOL if prec == "bf16" else FP32_OUT_TOL
    out = torch.empty(M, N, device="cuda", dtype=dt)
    G.matmul_forward_fused(out, None, x, w, b, "bias", prec)
    assert norm_err(_f64(out), h) <= tol
    G.matmul_forward_fused(out, r, x, w, b, "residual", prec)
    assert norm_err(_f64(out), O.residual_forward(r64, h)) <= tol
    pre = torch.empty(M, N, device="cuda", dtype=dt)
    G.matmul_forward_fused(out, pre, x, w, b, "gelu", prec)
    G.layer_check()
    assert norm_err(_f64(pre), h) <= tol
    assert norm_err(_f64(out), O.gelu_forward(h)) <= (GELU_TOL if prec == "bf16" else FP32_OUT_TOL)
    # the GELU backward: dinp (M, N) = (dy (M, K) W (K, N)) * gelu'(p), p drawn apart
    g = torch.Generator(device="cuda")
    g.manual_seed(M * N)
    dy = torch.randn(M, K, device="cuda", generator=g).to(dt)
    w2 = (torch.randn(K, N, device="cuda", generator=g) / np.sqrt(K)).to(dt)
    p = (1.5 * torch.randn(M, N, device="cuda", generator=g)).to(dt)
    dinp = torch.empty(M, N, device="cuda", dtype=dt)
    dbias = torch.zeros(N, device="cuda")
    sc = torch.empty(G.matmul_backward_input_gelu_scratch_bytes(M, N), dtype=torch.uint8, device="cuda")
    G.matmul_backward_input_gelu(dinp, dy, w2, p, prec, dbias, sc)
    G.layer_check()
    ref = O.gelu_backward(_f64(dy) @ _f64(w2), _f64(p))
    assert norm_err(_f64(dinp), ref) <= (GELU_BWD_TOL if prec == "bf16" else FP32_OUT_TOL)
    # bias gradient: the stored dinp's column sums (ragged row blocks and columns)
    assert norm_err(dbias.double().cpu().numpy(), _f64(dinp).sum(axis=0)) <= FP32_OUT_TOL


def test_bf16_shapes_off_the_tensor_core_path_are_refused(G):
    """bf16 runs on the tensor cores only: a product whose N or K is not a multiple of 8
    is refused (GPT2_EUNSUPPORTED), never sent to a slower kernel."""
    import torch
    bf = torch.bfloat16
    x = torch.zeros(64, 60, device="cuda", dtype=bf)
    w = torch.zeros(64, 60, device="cuda", dtype=bf)
    out = torch.empty(64, 64, device="cuda", dtype=bf)
    with pytest.raises(G.GPT2Error) as e:
        G.matmul_forward(out, x, w, None, "bf16")
    assert e.value.status == 8
    x = torch.zeros(64, 64, device="cuda", dtype=bf)
    w = torch.zeros(60, 64, device="cuda", dtype=bf)
    out = torch.empty(64, 60, device="cuda", dtype=bf)
    with pytest.raises(G.GPT2Error) as e:
        G.matmul_forward(out, x, w, None, "bf16")
    assert e.value.status == 8
    # and attention in bf16 takes head size 64 only
    qkv = torch.zeros(1, 16, 3 * 64, device="cuda", dtype=bf)
    o = torch.empty(1, 16, 64, device="cuda", dtype=bf)
    lse = torch.empty(1, 4, 16, device="cuda")
    with pytest.raises(G.GPT2Error) as e:
        G.attention_forward(o, lse, qkv, 4, "bf16")
    assert e.value.status == 8
