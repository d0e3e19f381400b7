"""Per-layer parity: the CUDA kernels through the C ABI against the CPU oracle (fp64)."""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from step_gpt_train_03_b300 import synth
from tests.gpu_helpers import ensure_built, norm_err

pytestmark = pytest.mark.gpu

# fp32 tolerances: outputs 1e-5 (a few fp32 roundings of O(1) values), gradients 1e-3
# normalised max-abs (the fp32-path bar of the training-step spec).
OUT_TOL = 1e-5
GRAD_TOL = 1e-3


@pytest.fixture(scope="module")
def L():
    ensure_built()
    import torch
    from step_gpt_train_03_b300 import gpt2lib
    torch.cuda.init()
    return gpt2lib


def _ln_case(L, N, C, seed=2):
    import torch
    x, w, b, dy = synth.layernorm_inputs(N, C, seed)
    dev = lambda a: torch.as_tensor(a).cuda()
    out = torch.empty((N, C), device="cuda")
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    L.layernorm_forward(out, mean, rstd, dev(x), dev(w), dev(b))
    dinp0 = np.random.default_rng(9).standard_normal((N, C)).astype(np.float32)
    dinp = dev(dinp0.copy())
    dw = torch.zeros(C, device="cuda")
    db = torch.zeros(C, device="cuda")
    scratch = torch.empty(max(L.layernorm_backward_scratch_bytes(N, C), 4), dtype=torch.uint8, device="cuda")
    L.layernorm_backward(dinp, dw, db, dev(dy), dev(x), dev(w), mean, rstd, scratch)
    torch.cuda.synchronize()
    x64, w64, b64, dy64 = (a.astype(np.float64) for a in (x, w, b, dy))
    y_ref, m_ref, r_ref = O.layernorm_forward(x64, w64, b64)
    dx_ref, dw_ref, db_ref = O.layernorm_backward(dy64, x64, w64, m_ref, r_ref)
    errs = {
        "y": norm_err(out.cpu().numpy(), y_ref),
        "mean": norm_err(mean.cpu().numpy(), m_ref),
        "rstd": norm_err(rstd.cpu().numpy(), r_ref),
        "dx": norm_err(dinp.cpu().numpy() - dinp0, dx_ref),
        "dw": norm_err(dw.cpu().numpy(), dw_ref),
        "db": norm_err(db.cpu().numpy(), db_ref),
    }
    return errs


def test_layernorm_standalone_workload(L):
    """The standalone layernorm workload: x (8192, 768) ~ 3 N(0,1) + 0.5, fp32."""
    e = _ln_case(L, 8192, 768)
    for k in ("y", "mean", "rstd"):
        assert e[k] < OUT_TOL, e
    for k in ("dx", "dw", "db"):
        assert e[k] < GRAD_TOL, e
    assert max(e["dx"], e["dw"], e["db"]) < 1e-5, e     # well inside the bar


# (8000, 256) and (20000, 128): several rows per warp through the backward's pipelined
# (shared-memory staged) form, so every stage is reused and every barrier phase flips
@pytest.mark.parametrize("N,C", [(1, 768), (13, 768), (8191, 768), (5, 8), (33, 64), (100, 2048), (7, 1000),
                                 (8000, 256), (20000, 128)])
def test_layernorm_edge_shapes(L, N, C):
    e = _ln_case(L, N, C)
    for k in ("y", "mean", "rstd"):
        assert e[k] < OUT_TOL, e
    for k in ("dx", "dw", "db"):
        assert e[k] < GRAD_TOL, e


def test_layernorm_empty_and_invalid(L):
    import torch
    z = torch.empty(0, device="cuda")
    L.layernorm_forward(z, z, z, torch.empty((0, 64), device="cuda"), torch.ones(64, device="cuda"),
                        torch.zeros(64, device="cuda"))
    with pytest.raises(L.GPT2Error):
        x = torch.zeros((4, 12), device="cuda")          # C not a multiple of 8
        L.layernorm_forward(x, torch.zeros(4, device="cuda"), torch.zeros(4, device="cuda"), x,
                            torch.ones(12, device="cuda"), torch.zeros(12, device="cuda"))


def _mm_case(L, M, N, K, precision, seed=0):
    import torch
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (0.1 * rng.standard_normal((N, K))).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    dy = rng.standard_normal((M, N)).astype(np.float32)
    tdt = torch.float32 if precision == "fp32" else torch.bfloat16
    dev = lambda a: torch.as_tensor(a).cuda().to(tdt)
    xd, wd, bd, dyd = dev(x), dev(w), dev(b), dev(dy)
    # the oracle sees exactly the values the kernel sees
    x64, w64, b64, dy64 = (t.float().cpu().numpy().astype(np.float64) for t in (xd, wd, bd, dyd))
    out = torch.empty((M, N), device="cuda", dtype=tdt)
    L.matmul_forward(out, xd, wd, bd, precision)
    dinp = torch.empty((M, K), device="cuda", dtype=tdt)
    dW0 = rng.standard_normal((N, K)).astype(np.float32)
    dW = torch.as_tensor(dW0.copy()).cuda()
    dB = torch.zeros(N, device="cuda")
    scratch = torch.empty(L.matmul_backward_scratch_bytes(M, N), dtype=torch.uint8, device="cuda")
    L.matmul_backward(dinp, dW, dB, dyd, xd, wd, precision, scratch)
    torch.cuda.synchronize()
    y_ref = O.matmul_forward(x64, w64, b64)
    dx_ref, dw_ref, db_ref = O.matmul_backward(dy64, x64, w64)
    return {
        "y": norm_err(out.float().cpu().numpy(), y_ref),
        "dx": norm_err(dinp.float().cpu().numpy(), dx_ref),
        "dw": norm_err(dW.cpu().numpy() - dW0, dw_ref),
        "db": norm_err(dB.cpu().numpy(), db_ref),
    }


# fp32 shapes reach every form of the FMA product: 64 x 64 tiles (few tiles, no split),
# 128 x 128 tiles with 16-byte or scalar loads, with and without a split contraction
# (1000 x 768 x 768 and 300 x 1030 x 516 split the input and weight gradients;
# 2100 x 1300 x 130 runs the forward on 128 x 128 tiles with scalar loads, unsplit)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (64, 64, 64), (257, 130, 72), (1000, 768, 768),
                                   (300, 1030, 516), (2100, 1300, 130)])
def test_matmul_fp32(L, M, N, K):
    e = _mm_case(L, M, N, K, "fp32")
    assert max(e.values()) < OUT_TOL, e


def test_matmul_fp32_split_is_deterministic(L):
    """The split contraction adds its partials in a fixed order: two runs agree bit for bit."""
    import torch
    M, N, K = 300, 1030, 516
    g = torch.Generator().manual_seed(3)
    x = torch.randn(M, K, generator=g).cuda()
    w = torch.randn(N, K, generator=g).cuda()
    dy = torch.randn(M, N, generator=g).cuda()
    scratch = torch.empty(L.matmul_backward_scratch_bytes(M, N), dtype=torch.uint8, device="cuda")
    runs = []
    for _ in range(2):
        dx = torch.empty(M, K, device="cuda")
        dW = torch.zeros(N, K, device="cuda")
        dB = torch.zeros(N, device="cuda")
        L.matmul_backward(dx, dW, dB, dy, x, w, "fp32", scratch)
        torch.cuda.synchronize()
        runs.append((dx.cpu(), dW.cpu()))
    assert torch.equal(runs[0][0], runs[1][0]) and torch.equal(runs[0][1], runs[1][1])


# bf16: fp32 accumulation of exact bf16 products, output rounded to bf16 (relative 2^-9),
# so a normalised error of 1e-2 bounds the rounding of the stored result.
BF16_TOL = 1e-2


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (256, 2304, 768), (300, 200, 136), (16384, 768, 64),
                                   (128, 50304, 768), (1, 64, 64)])
def test_matmul_bf16(L, M, N, K):
    e = _mm_case(L, M, N, K, "bf16")
    assert e["y"] < BF16_TOL and e["dx"] < BF16_TOL, e
    assert e["dw"] < 1e-4 and e["db"] < 1e-4, e      # fp32 outputs: only the products' order differs


# bf16 attention: inputs are bf16, P is rounded to bf16 before P V and outputs are
# stored in bf16, so 2e-2 of the tensor's max bounds the rounding; LSE is fp32 math on
# bf16 scores (abs 2e-2).
ATT_TOL = 2e-2


@pytest.mark.parametrize("B,T,NH,C,precision", [(2, 64, 4, 256, "bf16"), (1, 200, 2, 128, "bf16"),
                                                (2, 1024, 12, 768, "bf16"), (3, 37, 2, 128, "bf16"),
                                                (2, 131, 1, 64, "bf16"), (1, 1, 1, 64, "bf16"),
                                                (2, 40, 4, 64, "fp32"), (1, 129, 2, 128, "fp32"),
                                                (1, 70, 1, 128, "fp32"), (2, 33, 1, 8, "fp32")])
def test_attention_forward_backward(L, B, T, NH, C, precision):
    import torch
    rng = np.random.default_rng(B * 1000 + T)
    qkv = rng.standard_normal((B, T, 3 * C)).astype(np.float32)
    dout = rng.standard_normal((B, T, C)).astype(np.float32)
    tdt = torch.bfloat16 if precision == "bf16" else torch.float32
    qkv_d = torch.as_tensor(qkv).cuda().to(tdt)
    dout_d = torch.as_tensor(dout).cuda().to(tdt)
    q64 = qkv_d.float().cpu().numpy().astype(np.float64)
    d64 = dout_d.float().cpu().numpy().astype(np.float64)
    out = torch.empty((B, T, C), device="cuda", dtype=tdt)
    lse = torch.empty((B, NH, T) if precision == "bf16" else (B, NH, T, T), device="cuda")
    L.attention_forward(out, lse, qkv_d, NH, precision)
    dqkv = torch.empty_like(qkv_d)
    scratch = torch.empty(L.attention_backward_scratch_bytes(B, T, C, NH, precision), dtype=torch.uint8,
                          device="cuda")
    db0 = torch.as_tensor(rng.standard_normal(3 * C).astype(np.float32)).cuda()
    dbias = db0.clone()
    L.attention_backward(dqkv, dout_d, qkv_d, out, lse, NH, precision, scratch, dbias)
    torch.cuda.synchronize()
    ref_out, pre, att = O.attention_forward(q64, NH)
    ref_dqkv = O.attention_backward(d64, q64, att, NH)
    tol = ATT_TOL if precision == "bf16" else OUT_TOL
    assert norm_err(out.float().cpu().numpy(), ref_out) < tol
    got_dqkv = dqkv.float().cpu().numpy().astype(np.float64)
    assert norm_err(got_dqkv, ref_dqkv) < (tol if precision == "bf16" else GRAD_TOL)
    # the qkv bias gradient added into dbias: the stored dqkv's column sums (exact up to
    # fp32 summation), and the oracle's within the dqkv tolerance
    db = (dbias - db0).double().cpu().numpy()
    assert norm_err(db, got_dqkv.reshape(-1, 3 * C).sum(axis=0)) < 1e-5
    assert norm_err(db, ref_dqkv.reshape(-1, 3 * C).sum(axis=0)) < (tol if precision == "bf16" else GRAD_TOL)
    if precision == "bf16":
        m = pre.max(-1, keepdims=True)
        ref_lse = (m + np.log(np.exp(pre - m).sum(-1, keepdims=True)))[..., 0]
        assert np.abs(lse.cpu().numpy() - ref_lse).max() < 2e-2
