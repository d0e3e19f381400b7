"""gpt2_layernorm_backward_noalloc: the layernorm backward for callers that cannot
allocate device memory (a host program that passes only its input and output buffers,
or one whose device memory is all committed at start-up).  It must give the same
results as gpt2_layernorm_backward with a caller-provided scratch buffer, call after
call, although every call reuses the same built-in scratch array.

This file is named so that pytest collects it last."""
import numpy as np
import pytest

from step_gpt_train_03_b300 import synth
from tests.gpu_helpers import ensure_built, norm_err

pytestmark = pytest.mark.gpu

# the tolerances of the other fp32 layernorm tests: 1e-3 normalised max-abs for gradients
GRAD_TOL = 1e-3


def _inputs(N, C, seed):
    import torch
    from step_gpt_train_03_b300 import gpt2lib as G
    x, w, b, dy = (torch.as_tensor(a).cuda() for a in synth.layernorm_inputs(N, C, seed))
    out = torch.empty((N, C), device="cuda")
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    G.layernorm_forward(out, mean, rstd, x, w, b)
    dinp0 = torch.as_tensor(np.random.default_rng(seed + 1).standard_normal((N, C)).astype(np.float32)).cuda()
    return x, w, dy, mean, rstd, dinp0


def _run(fn, x, w, dy, mean, rstd, dinp0, **kw):
    import torch
    dinp = dinp0.clone()
    dw = torch.zeros(x.shape[1], device="cuda")
    db = torch.zeros(x.shape[1], device="cuda")
    fn(dinp, dw, db, dy, x, w, mean, rstd, **kw)
    torch.cuda.synchronize()
    return dinp.cpu().numpy(), dw.cpu().numpy(), db.cpu().numpy()


def test_noalloc_layernorm_backward_matches_allocating_entry_point():
    ensure_built()
    import torch
    from step_gpt_train_03_b300 import gpt2lib as G
    # calls in a row, of different shapes, so stale scratch from an earlier call would
    # show; (4096, 2048) is the largest shape accepted at C = 2048 (its partial sums fill
    # the array exactly) and runs the shared-memory pipelined kernel with one block per SM
    for N, C, seed in ((8192, 768, 2), (1000, 1024, 5), (4096, 2048, 7), (8192, 768, 2)):
        args = _inputs(N, C, seed)
        scratch = torch.empty(G.layernorm_backward_scratch_bytes(N, C), dtype=torch.uint8, device="cuda")
        ref = _run(G.layernorm_backward, *args, scratch=scratch)
        got = _run(G.layernorm_backward_noalloc, *args)
        G.layer_check()
        for r, g in zip(ref, got):
            assert norm_err(g, r) <= GRAD_TOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ensure_built()
    import torch
    from step_gpt_train_03_b300 import gpt2lib as G
    # at C = 2048 the partials take min(ceil(N / 16), 296) blocks x 2C floats: 4 MiB at
    # N = 4096 (accepted above), 4 MiB + 16 KiB at N = 4097, 4.625 MiB (296 blocks) from
    # N = 4721 on
    for N in (4097, 32768):
        C = 2048
        assert G.layernorm_backward_scratch_bytes(N, C) > G.NOALLOC_SCRATCH_BYTES
        t = torch.zeros((N, C), device="cuda")
        v = torch.zeros(C, device="cuda")
        r = torch.ones(N, device="cuda")
        with pytest.raises(G.GPT2Error) as e:
            G.layernorm_backward_noalloc(t, v.clone(), v.clone(), t, t, v, r, r)
        assert e.value.status == 1
    assert G.layernorm_backward_scratch_bytes(4096, 2048) == G.NOALLOC_SCRATCH_BYTES
