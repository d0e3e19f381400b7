"""The rows after the training step, through the C ABI against the oracle: forward-only
evaluation, next-token sampling (and generation), parameter files.

The llm.c article's training run evaluates a validation loss, generates samples from
the model after training, and starts from a weight checkpoint written for the C
program; the sampler (inverse CDF driven by SplitMix64) and the file layout are this
library's readings, restated independently by the oracle."""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from step_gpt_train_03_b300 import synth
from tests.gpu_helpers import dev_tokens, ensure_built, gpu_model
from tests.oracle_helpers import make_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    import torch
    torch.cuda.init()


def _check_draws(got, logits, V, temperature, seed, tol):
    """Each GPU token is the oracle's draw, or (the logits differ by rounding) the oracle's
    threshold lies within tol * total of that token's interval of the running sum."""
    for b, k in enumerate(got):
        kk, lo, hi, thr, tot = O.sample_token(logits[b], V, temperature, seed, b)
        assert 0 <= k < V
        if k != kk:
            x = logits[b][:V].astype(np.float64)
            c = np.cumsum(np.exp((x - x.max()) / temperature))
            lo_k = 0.0 if k == 0 else float(c[k - 1])
            assert lo_k - tol * tot <= thr <= float(c[k]) + tol * tot, (b, int(k), kk)


def test_sampling_fp32_matches_oracle():
    shape = synth.TINY
    B, T = 8, 32
    tok, _ = synth.uniform_tokens(512, B, T, 7)
    m = gpu_model(shape, B, T, "fp32", 0)
    o = make_oracle(shape, 0)
    m.forward(dev_tokens(tok), None, want_loss=False)
    o.forward(tok)
    logits = o.acts["logits"]
    for pos, temp, seed in ((T - 1, 1.0, 42), (5, 0.7, 9), (0, 1.5, 2 ** 63 + 5)):
        got = m.sample(pos, temp, seed).cpu().numpy()
        _check_draws(got, logits[:, pos, :], 512, temp, seed, 1e-5)
    a = m.sample(T - 1, 1.0, 42).cpu().numpy()
    b = m.sample(T - 1, 1.0, 42).cpu().numpy()
    assert (a == b).all()                                    # a seed always gives the same tokens


def test_sampling_bf16_124m_within_rounding():
    shape = synth.GPT2_124M
    B, T = 4, 64
    tok, _ = synth.zipf_batches(shape.vocab_size, B, T, 1, 8)[0]
    m = gpu_model(shape, B, T, "bf16", 2)
    o = make_oracle(shape, 2)
    m.forward(dev_tokens(tok), None, want_loss=False)
    o.forward(tok)
    got = m.sample(T - 1, 1.0, 1234).cpu().numpy()
    _check_draws(got, o.acts["logits"][:, T - 1, :], shape.vocab_size, 1.0, 1234, 2e-2)


def test_sampling_needs_kept_logits_and_valid_arguments():
    from step_gpt_train_03_b300.gpt2lib import GPT2Error
    m = gpu_model(synth.TINY, 2, 32, "fp32", 0)
    tok, tgt = synth.uniform_tokens(512, 2, 32, 1)
    m.forward(dev_tokens(tok), dev_tokens(tgt))              # the logits became d loss / d logits
    with pytest.raises(GPT2Error) as e:
        m.sample(31, 1.0, 1)
    assert e.value.status == 2
    m.forward(dev_tokens(tok), None, want_loss=False)
    for pos, temp in ((32, 1.0), (-1, 1.0), (3, 0.0), (3, -1.0)):
        with pytest.raises(GPT2Error) as e:
            m.sample(pos, temp, 1)
        assert e.value.status == 1


def test_generate_extends_the_prompt_with_sampled_tokens():
    import torch
    m = gpu_model(synth.TINY, 2, 32, "fp32", 0)
    prompt = dev_tokens(synth.uniform_tokens(512, 2, 4, 3)[0])
    out = m.generate(prompt, 6, 1.0, 99)
    assert out.shape == (2, 10)
    assert torch.equal(out[:, :4], prompt)
    assert int(out.min()) >= 0 and int(out.max()) < 512
    m.forward(prompt, None, want_loss=False)
    assert torch.equal(m.sample(3, 1.0, 99), out[:, 4])


def test_eval_loss_matches_oracle():
    """Forward-only evaluation (no backward, no update): the mean loss of a batch."""
    shape = synth.TINY
    tok, tgt = synth.uniform_tokens(512, 2, 32, 11)
    m = gpu_model(shape, 2, 32, "fp32", 0)
    o = make_oracle(shape, 0)
    loss = m.forward(dev_tokens(tok), dev_tokens(tgt))
    ref = o.forward(tok, tgt)
    assert abs(loss - ref) <= 1e-5 * abs(ref)


def test_param_file_round_trip(tmp_path):
    import torch
    shape = synth.TINY
    a = gpu_model(shape, 2, 32, "fp32", 0)
    path = tmp_path / "w.bin"
    a.save(path)
    h, tensors = O.read_param_file(path)
    assert h[0] == O.PARAM_FILE_MAGIC and h[1] == O.PARAM_FILE_VERSION
    assert [int(x) for x in h[2:8]] == [32, 512, 2, 4, 64, 512] and not h[8:].any()
    ref = synth.init_params(shape, 0)
    for k in O.PARAM_ORDER:
        np.testing.assert_array_equal(tensors[k], np.asarray(ref[k], dtype=np.float32), err_msg=k)
    b = gpu_model(shape, 2, 32, "fp32", 5)                   # other weights, then the file's
    b.load(path)
    assert torch.equal(a.flat_params(), b.flat_params())
    # the oracle on the file's weights gives the loaded model's loss
    o = O.from_shape(shape)
    o.load({k: v.astype(np.float64) for k, v in tensors.items()})
    tok, tgt = synth.uniform_tokens(512, 2, 32, 4)
    ref_loss = o.forward(tok, tgt)
    assert abs(b.forward(dev_tokens(tok), dev_tokens(tgt)) - ref_loss) <= 1e-5 * abs(ref_loss)


def test_param_file_errors_leave_parameters_untouched(tmp_path):
    import torch
    from step_gpt_train_03_b300.gpt2lib import GPT2Error
    a = gpu_model(synth.TINY, 2, 32, "fp32", 0)
    good = tmp_path / "w.bin"
    a.save(good)
    other = gpu_model(synth.ModelShape(32, 512, 512, 3, 4, 64), 2, 32, "fp32", 1)   # three layers
    before = other.flat_params().clone()
    cut = tmp_path / "cut.bin"
    cut.write_bytes(good.read_bytes()[:5000])
    for target, path in ((other, good), (a, cut), (a, tmp_path / "missing.bin")):
        snap = target.flat_params().clone()
        with pytest.raises(GPT2Error) as e:
            target.load(path)
        assert e.value.status == 9
        assert torch.equal(target.flat_params(), snap)
    assert torch.equal(other.flat_params(), before)
