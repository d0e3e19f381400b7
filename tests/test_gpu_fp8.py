"""The fp8 variant (yinghuohong.cn llm.c article, section "脚动完成每一个层前向/反向流传":
precision taken from fp32 down to fp16 or lower) through the C ABI against the oracle.

Where floating point decides an e4m3 code, both sides decide it in fp32 on the same
values (weights), or on values that differ only by the layernorm's summation order
(activations), where a code may flip to its neighbour at a rounding midpoint.  The
products of e4m3 values are exact in fp32, so the tensor-core product is held to the
bf16 tolerance of its stored output against the oracle's exact product of the decoded
codes."""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from step_gpt_train_03_b300 import synth
from tests.gpu_helpers import dev_tokens, ensure_built, gpu_model, hp_of, norm_err, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

BF16_TOL = 4e-3            # stored-output rounding (2^-9) plus fp32 accumulation
GELU_TOL = 6e-3
LOSS_ABS = 2e-2            # as the bf16 path


@pytest.fixture(scope="module")
def G():
    ensure_built()
    import torch
    from step_gpt_train_03_b300 import gpt2lib
    torch.cuda.init()
    return gpt2lib


def test_weight_quantization_is_bit_exact(G):
    """Per-tensor e4m3 codes of fp32 weights equal the oracle's: both scale by the same
    power of two (exact) and round the same fp32 value to nearest even."""
    import torch
    rng = np.random.default_rng(0)
    for n, scale in ((768 * 2304, 0.02), (3072 * 768, 1.0), (1024, 300.0), (64, 1e-9)):
        x = (rng.standard_normal(n) * scale).astype(np.float32)
        xd = torch.as_tensor(x).cuda()
        codes = torch.empty(n, dtype=torch.uint8, device="cuda")
        deq = torch.empty(1, device="cuda")
        amax = torch.empty(1, dtype=torch.int32, device="cuda")
        G.quantize_e4m3(codes, deq, amax, xd)
        torch.cuda.synchronize()
        _, ref_codes, k = O.quantize_tensor_e4m3(x.astype(np.float64))
        assert np.array_equal(codes.cpu().numpy(), ref_codes), n
        assert deq.item() == 2.0 ** -k


@pytest.mark.parametrize("N,C", [(8192, 768), (37, 1024), (1, 64)])
def test_layernorm_fp8_output(G, N, C):
    """The layernorm's e4m3 row copy: every row's scale equals the oracle's, the codes
    equal the oracle's codes of its own (fp64) layernorm output except at rounding
    midpoints, where they may be the neighbouring code."""
    import torch
    x, w, b, _ = synth.layernorm_inputs(N, C, 2)
    dev = lambda a: torch.as_tensor(a).cuda()
    out = torch.empty((N, C), device="cuda")
    codes = torch.empty((N, C), dtype=torch.uint8, device="cuda")
    rdeq = torch.empty(N, device="cuda")
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    G.layernorm_forward_fp8(out, codes, rdeq, mean, rstd, dev(x), dev(w), dev(b))
    torch.cuda.synchronize()
    y, _, _ = O.layernorm_forward(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64))
    deq, ref_codes, ks = O.quantize_rows_e4m3(y)
    assert np.array_equal(rdeq.cpu().numpy(), np.exp2(-ks).astype(np.float32))
    got = codes.cpu().numpy()
    same = got == ref_codes
    assert same.mean() >= 0.999, same.mean()
    # where they differ, the two decoded values are neighbours on the e4m3 grid
    gv, rv = O.E4M3_TABLE[got[~same]], O.E4M3_TABLE[ref_codes[~same]]
    assert np.all(np.abs(gv - rv) <= 2.0 ** -3 * np.maximum(np.abs(gv), np.abs(rv)) + 2.0 ** -9)


def _rand_codes(rng, shape):
    """Random finite e4m3 codes (every code but the two NaNs)."""
    c = rng.integers(0, 254, shape).astype(np.uint8)
    return np.where(c >= 0x7F, c + 1, c).astype(np.uint8)      # skip 0x7F (and 0xFF)


@pytest.mark.parametrize("M,N,K,epi", [(16384, 2304, 768, "bias"), (16384, 3072, 768, "gelu"),
                                       (300, 264, 784, "bias"), (129, 520, 1040, "gelu")])
def test_fp8_matmul_against_exact_product(G, M, N, K, epi):
    """e4m3 codes with per-row and per-tensor power-of-two factors: the tensor-core
    product equals the oracle's exact product of the decoded values (then the epilogue)."""
    import torch
    rng = np.random.default_rng(M + N)
    a = _rand_codes(rng, (M, K))
    wc = _rand_codes(rng, (N, K))
    # factors that put the products at unit scale (so the bias does not dominate and the
    # GELU sees its whole curve): per-row 2^-6 .. 2^-8, weight 2^-11
    adeq = np.exp2(-rng.integers(6, 9, M)).astype(np.float32)
    wdeq = np.array([2.0 ** -11], np.float32)
    bias = (0.1 * rng.standard_normal(N)).astype(np.float32)
    bias_d = torch.as_tensor(bias).cuda().to(torch.bfloat16)
    out = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
    aux = torch.empty((M, N), device="cuda", dtype=torch.bfloat16) if epi == "gelu" else None
    G.matmul_forward_fp8(out, aux, torch.as_tensor(a).cuda(), torch.as_tensor(adeq).cuda(), torch.as_tensor(wc).cuda(),
                         torch.as_tensor(wdeq).cuda(), bias_d, epi)
    G.layer_check()
    A = O.E4M3_TABLE[a] * adeq[:, None].astype(np.float64)
    W = O.E4M3_TABLE[wc] * float(wdeq[0])
    h = O.matmul_forward(A, W, bias_d.float().cpu().numpy().astype(np.float64))
    if epi == "bias":
        assert norm_err(out.float().cpu().numpy(), h) <= BF16_TOL
    else:
        assert norm_err(aux.float().cpu().numpy(), h) <= BF16_TOL
        assert norm_err(out.float().cpu().numpy(), O.gelu_forward(h)) <= GELU_TOL


def test_model_weight_shadows_equal_the_oracle_quantization(G):
    """After loading the weights (and after an update) the fp8 model's e4m3 shadows of
    qkvw and fcw are the oracle's per-(tensor, layer) quantization of the fp32 masters."""
    shape = synth.TINY_HS64
    m = gpu_model(shape, 2, 32, "fp8", 0)
    tok, tgt = synth.uniform_tokens(shape.vocab_size, 2, 32, 0)
    for step in range(2):
        P = {k: v.detach().cpu().numpy() for k, v in m.params().items()}
        for name in ("qkvw", "fcw"):
            codes, deq = m.fp8_weights(name)
            codes, deq = codes.cpu().numpy(), deq.cpu().numpy()
            for l in range(shape.num_layers):
                _, ref, k = O.quantize_tensor_e4m3(P[name][l].astype(np.float64))
                assert np.array_equal(codes[l], ref), (step, name, l)
                assert deq[l] == 2.0 ** -k
        m.step(dev_tokens(tok), dev_tokens(tgt), 1e-3, 0.9, 0.95, 1e-8, 0.1, step + 1)


def test_fp8_tiny_ten_steps(G):
    shape = synth.TINY_HS64
    batches = synth.workload_batches(synth.WORKLOADS["tiny_fp32"], 10)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    _, lg, _ = run_gpu(shape, "fp8", 0, batches, hp)
    from tests.oracle_helpers import make_oracle
    o = make_oracle(shape, 0)
    o.fp8 = True
    lo = [o.step(*b, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], i + 1)
          for i, b in enumerate(batches)]
    assert max(abs(a - b) for a, b in zip(lg, lo)) <= LOSS_ABS, (lg, lo)


@pytest.mark.slow
def test_fp8_gpt2_124m_short_sequences_ten_steps(G):
    """124M shape in the fp8 mode (B=2, T=128, fresh Zipf batches, lr 6e-4, wd 0.1)
    against the oracle in its fp8 mode (fp32), every step within 2e-2."""
    shape = synth.GPT2_124M
    batches = synth.zipf_batches(50257, 2, 128, 10, 21)
    hp = dict(lr=6e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    _, lg, _ = run_gpu(shape, "fp8", 2, batches, hp)
    from tests.oracle_helpers import make_oracle
    o = make_oracle(shape, 2, np.float32)
    o.fp8 = True
    lo = [o.step(*b, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], i + 1)
          for i, b in enumerate(batches)]
    assert max(abs(a - b) for a, b in zip(lg, lo)) <= LOSS_ABS, (lg, lo)
