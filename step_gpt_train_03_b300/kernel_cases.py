"""Run one kernel of the training step on its own, at the 124M workload's sizes, a few
times: the target of per-kernel Nsight Compute captures.

    python -m step_gpt_train_03_b300.kernel_cases <case> [--iters N] [--time]

With --time, the runs are timed with CUDA events (after the untimed ones) and the
case's algorithmic work rate is printed (TFLOP/s for products, GB/s for layernorm).
With --flush, each timed run is bracketed by its own events and preceded (outside the
events) by a write of 256 MB, twice the 126 MB L2, so no input starts in L2 (the events
then also time the launch).  With --rotate (layernorm cases), the runs go back to back
over six copies of the per-row tensors, a working set larger than L2.

Cases (B*T = 16384 rows, C = 768, NH = 12, Vp = 50304, bf16 unless stated):
  matmul_fc_forward       (16384 x 768) @ (3072 x 768)^T
  matmul_lmhead_forward   (16384 x 768) @ (50304 x 768)^T
  matmul_lmhead_backward  dX (16384 x 768) and dW (50304 x 768, fp32 +=) of the LM head
  attention_forward       causal, B=16, T=1024, hs=64
  attention_backward      same sizes (dK/dV kernel, then dQ kernel)
  layernorm_forward_fp32  (8192 x 768) fp32, the standalone layernorm workload
  layernorm_backward_fp32 the same workload's backward
  eval_124m               forward-only evaluation of GPT-2 124M (bf16, B=16, T=1024, loss)
  sample_124m             next-token sampling over the 16 rows of that forward's logits
"""
from __future__ import annotations

import argparse
import sys


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--time", action="store_true")
    ap.add_argument("--flush", action="store_true")
    ap.add_argument("--rotate", action="store_true")
    args = ap.parse_args(argv)
    import torch
    from step_gpt_train_03_b300 import gpt2lib as G
    torch.manual_seed(0)
    BT, C, NH, Vp, B, T = 16384, 768, 12, 50304, 16, 1024
    dev = "cuda"
    bf = torch.bfloat16
    case = args.case
    if case.startswith("matmul"):
        N = 3072 if case == "matmul_fc_forward" else Vp
        x = torch.randn(BT, C, device=dev).to(bf)
        w = (0.02 * torch.randn(N, C, device=dev)).to(bf)
        work, unit = 2.0 * BT * N * C, "flop"
        if case.endswith("forward"):
            out = torch.empty(BT, N, device=dev, dtype=bf)
            run = lambda: G.matmul_forward(out, x, w, None, "bf16")
        else:
            dy = (1e-4 * torch.randn(BT, N, device=dev)).to(bf)
            dx = torch.empty(BT, C, device=dev, dtype=bf)
            dW = torch.zeros(N, C, device=dev)
            sc = torch.empty(G.matmul_backward_scratch_bytes(BT, N), dtype=torch.uint8, device=dev)
            run = lambda: G.matmul_backward(dx, dW, None, dy, x, w, "bf16", sc)
            work = 2 * work                                # dX and dW
    elif case.startswith("attention"):
        qkv = torch.randn(B, T, 3 * C, device=dev).to(bf)
        out = torch.empty(B, T, C, device=dev, dtype=bf)
        lse = torch.empty(B, NH, T, device=dev)
        G.attention_forward(out, lse, qkv, NH, "bf16")
        work, unit = 4.0 * B * C * T * (T + 1) / 2, "flop"       # Q K^T and P V over the causal half
        if case == "attention_forward":
            run = lambda: G.attention_forward(out, lse, qkv, NH, "bf16")
        else:
            dout = torch.randn(B, T, C, device=dev).to(bf)
            dqkv = torch.empty_like(qkv)
            sc = torch.empty(G.attention_backward_scratch_bytes(B, T, C, NH, "bf16"), dtype=torch.uint8, device=dev)
            run = lambda: G.attention_backward(dqkv, dout, qkv, out, lse, NH, "bf16", sc)
            work = 2 * work                                # dP, dV, dK, dQ (recomputed S not counted)
    elif case in ("layernorm_backward_fp32", "layernorm_forward_fp32"):
        N = 8192
        x = 3 * torch.randn(N, C, device=dev) + 0.5
        w = 1 + 0.1 * torch.randn(C, device=dev)
        b = 0.1 * torch.randn(C, device=dev)
        dy = torch.randn(N, C, device=dev)
        y = torch.empty_like(x)
        mean = torch.empty(N, device=dev)
        rstd = torch.empty(N, device=dev)
        G.layernorm_forward(y, mean, rstd, x, w, b)
        dx = torch.zeros_like(x)
        dw = torch.zeros(C, device=dev)
        db = torch.zeros(C, device=dev)
        sc = torch.empty(G.layernorm_backward_scratch_bytes(N, C), dtype=torch.uint8, device=dev)
        # --rotate: six copies of every per-row tensor (6 x 4 x 25 MB > the 126 MB L2), used
        # in turn, so back-to-back runs never find their inputs in L2
        ncopy = 6 if args.rotate else 1
        X = [x] + [x.clone() for _ in range(ncopy - 1)]
        Y = [y] + [torch.empty_like(y) for _ in range(ncopy - 1)]
        DY = [dy] + [dy.clone() for _ in range(ncopy - 1)]
        DX = [dx] + [torch.zeros_like(dx) for _ in range(ncopy - 1)]
        ST = [(mean, rstd)] + [(torch.empty_like(mean), torch.empty_like(rstd)) for _ in range(ncopy - 1)]
        for i in range(1, ncopy):
            G.layernorm_forward(Y[i], ST[i][0], ST[i][1], X[i], w, b)
        ctr = [0]

        def pick():
            i = ctr[0] % ncopy
            ctr[0] += 1
            return i
        if case == "layernorm_backward_fp32":
            def run():
                i = pick()
                G.layernorm_backward(DX[i], dw, db, DY[i], X[i], w, ST[i][0], ST[i][1], sc)
            work, unit = 4.0 * N * C * 4 + 8.0 * N, "byte"     # dy, x, dinp read; dinp written; stats
        else:
            def run():
                i = pick()
                G.layernorm_forward(Y[i], ST[i][0], ST[i][1], X[i], w, b)
            work, unit = 2.0 * N * C * 4 + 8.0 * N, "byte"     # x read, y written; stats
    elif case in ("eval_124m", "sample_124m"):
        from step_gpt_train_03_b300 import synth
        w = synth.WORKLOADS["gpt2_124m_bf16_b16_t1024"]
        m = G.GPT2(w.shape, B, T, "bf16")
        m.load_params(synth.init_params(w.shape, w.seed))
        tok, tgt = synth.zipf_batches(w.shape.vocab_size, B, T, 1, w.seed)[0]
        tok = torch.as_tensor(tok).to(dev)
        tgt = torch.as_tensor(tgt).to(dev)
        if case == "eval_124m":
            run = lambda: m.forward(tok, tgt, want_loss=False)
            work, unit = float(B * T), "token"
        else:
            m.forward(tok, None, want_loss=False)
            outk = torch.empty(B, dtype=torch.int32, device=dev)
            run = lambda: m.sample(T - 1, 1.0, 7, outk)
            work, unit = float(B), "token"
    else:
        print(f"unknown case {case}", file=sys.stderr)
        return 2
    for _ in range(args.iters):
        run()
    torch.cuda.synchronize()
    print(f"{case}: {args.iters} runs ok")
    if args.time:
        if args.flush:
            junk = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
            total = 0.0
            for _ in range(args.iters):
                junk.fill_(1)
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record()
                run()
                e.record()
                e.synchronize()
                total += s.elapsed_time(e)
            sec = total / 1e3 / args.iters
        else:
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(args.iters):
                run()
            e.record()
            e.synchronize()
            sec = s.elapsed_time(e) / 1e3 / args.iters
        rate = (f"{work / sec / 1e12:.1f} TFLOP/s" if unit == "flop" else
                f"{work / sec / 1e9:.0f} GB/s" if unit == "byte" else f"{work / sec:.0f} tokens/s")
        print(f"{case}: {sec * 1e6:.1f} us per run, {rate} (algorithmic){', L2 flushed' if args.flush else ', 6 rotating input copies' if args.rotate else ''}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
