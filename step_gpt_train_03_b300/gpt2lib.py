"""Python binding of the C ABI in include/gpt2.h (ctypes; argument marshalling only).

Every step of the training path runs in the CUDA library libgpt2_b300.so.  PyTorch is
used for device memory (one uint8 workspace tensor) and the CUDA stream.  If the library
has not been built the import of this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgpt2_b300.so")

FP32, BF16, FP8 = 0, 1, 2
PRECISIONS = {"fp32": FP32, "bf16": BF16, "fp8": FP8}
STATUS = {0: "GPT2_OK", 1: "GPT2_EINVAL", 2: "GPT2_ESTATE", 3: "GPT2_ECUDA", 4: "GPT2_ETOKEN",
          5: "GPT2_ENONFINITE", 6: "GPT2_ETIMEOUT", 7: "GPT2_ENOMEM", 8: "GPT2_EUNSUPPORTED",
          9: "GPT2_EIO"}
PARAM_ORDER = ("wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
               "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb")

# exported symbols and their signatures (restype, argtypes)
_vp, _i, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_psz = ctypes.POINTER(ctypes.c_size_t)


class GPT2Config(ctypes.Structure):
    _fields_ = [("max_seq_len", _i), ("vocab_size", _i), ("padded_vocab_size", _i),
                ("num_layers", _i), ("num_heads", _i), ("channels", _i)]


SIGNATURES = {
    "gpt2_workspace_bytes": (_i, [ctypes.POINTER(GPT2Config), _i, _i, _i, _psz]),
    "gpt2_build": (_i, [ctypes.POINTER(GPT2Config), _i, _i, _i, _vp, _sz, _vp, ctypes.POINTER(_vp)]),
    "gpt2_free": (None, [_vp]),
    "gpt2_destroy": (None, [_vp]),
    "gpt2_num_params": (_i, [_vp, _psz]),
    "gpt2_param_ptr": (_i, [_vp, ctypes.POINTER(_vp)]),
    "gpt2_grad_ptr": (_i, [_vp, ctypes.POINTER(_vp)]),
    "gpt2_layer_check": (_i, [_vp]),
    "gpt2_update_muon": (_i, [_vp, _f, _f, _i, _f, _f, _f, _f, _f, _i]),
    "gpt2_newton_schulz_scratch_bytes": (_sz, [_i, _i]),
    "gpt2_newton_schulz": (_i, [_vp, _vp, _i, _i, _i, _vp, _sz, _vp]),
    "gpt2_layernorm_forward_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp]),
    "gpt2_quantize_e4m3": (_i, [_vp, _vp, _vp, _vp, _sz, _vp]),
    "gpt2_matmul_forward_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "gpt2_fp8_weights": (_i, [_vp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp)]),
    "gpt2_matmul_forward_fused": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "gpt2_matmul_backward_input_gelu_scratch_bytes": (_sz, [_i, _i]),
    "gpt2_matmul_backward_input_gelu": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp]),
    "gpt2_set_stream": (_i, [_vp, _vp]),
    "gpt2_num_parameters": (_i, [_vp, _psz, _psz]),
    "gpt2_param_tensor": (_i, [_vp, _i, _psz, _psz]),
    "gpt2_params": (_vp, [_vp]),
    "gpt2_grads": (_vp, [_vp]),
    "gpt2_adam_m": (_vp, [_vp]),
    "gpt2_adam_v": (_vp, [_vp]),
    "gpt2_sync_params": (_i, [_vp]),
    "gpt2_forward": (_i, [_vp, _vp, _vp, _i, _i, ctypes.POINTER(_f)]),
    "gpt2_zero_grad": (_i, [_vp]),
    "gpt2_backward": (_i, [_vp]),
    "gpt2_update": (_i, [_vp, _f, _f, _f, _f, _f, _i]),
    "gpt2_step_host": (_i, [_vp, _vp, _vp, _i, _i, _f, _f, _f, _f, _f, _i, ctypes.POINTER(_f)]),
    "gpt2_step": (_i, [_vp, _vp, _vp, _i, _i, _f, _f, _f, _f, _f, _i, ctypes.POINTER(_f)]),
    "gpt2_step_muon": (_i, [_vp, _vp, _vp, _i, _i, _f, _f, _i, _f, _f, _f, _f, _f, _i, ctypes.POINTER(_f)]),
    "gpt2_set_graphs": (_i, [_vp, _i]),
    "gpt2_sample": (_i, [_vp, _i, _f, ctypes.c_ulonglong, _vp]),
    "gpt2_save_params": (_i, [_vp, ctypes.c_char_p]),
    "gpt2_load_params": (_i, [_vp, ctypes.c_char_p]),
    "gpt2_loss": (_vp, [_vp]),
    "gpt2_losses": (_vp, [_vp]),
    "gpt2_logits": (_vp, [_vp]),
    "gpt2_check": (_i, [_vp]),
    "gpt2_strerror": (ctypes.c_char_p, [_i]),
    "gpt2_last_cuda_error": (_i, []),
    "gpt2_kernel_launches": (ctypes.c_longlong, []),
    "gpt2_profile_enable": (_i, [ctypes.c_uint]),
    "gpt2_profile_collect": (_i, []),
    "gpt2_profile_reset": (_i, []),
    "gpt2_profile_read": (_i, [_i, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong),
                               ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
    "gpt2_profile_dropped": (ctypes.c_longlong, []),
    "gpt2_profile_num_classes": (_i, []),
    "gpt2_profile_class_name": (ctypes.c_char_p, [_i]),
    "gpt2_layernorm_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp]),
    "gpt2_layernorm_backward_scratch_bytes": (_sz, [_i, _i]),
    "gpt2_layernorm_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp, _sz, _vp]),
    "gpt2_layernorm_backward_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp]),
    "gpt2_attention_forward": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "gpt2_attention_backward_scratch_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "gpt2_attention_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "gpt2_matmul_forward": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "gpt2_matmul_backward_scratch_bytes": (_sz, [_i, _i]),
    "gpt2_matmul_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _sz, _vp]),
}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} (run python -m step_gpt_train_03_b300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = load_library()


class GPT2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.gpt2_strerror(status).decode()
        extra = ""
        if status == 3:
            extra = f" (cudaError {lib.gpt2_last_cuda_error()})"
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}{extra}")


def check(status: int, where: str) -> None:
    if status != 0:
        raise GPT2Error(status, where)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream_handle(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def config_of(shape) -> GPT2Config:
    return GPT2Config(shape.max_seq_len, shape.vocab_size, shape.padded_vocab_size,
                      shape.num_layers, shape.num_heads, shape.channels)


def workspace_bytes(shape, max_B: int, max_T: int, precision: str) -> int:
    n = ctypes.c_size_t(0)
    cfg = config_of(shape)
    check(lib.gpt2_workspace_bytes(ctypes.byref(cfg), max_B, max_T, PRECISIONS[precision],
                                   ctypes.byref(n)), "gpt2_workspace_bytes")
    return n.value


class GPT2:
    """One model on one GPU: a torch uint8 workspace carved by gpt2_build."""

    def __init__(self, shape, max_B: int, max_T: int, precision: str = "bf16", device="cuda",
                 stream=None):
        import torch
        self.shape = shape
        self.precision = precision
        self.max_B, self.max_T = max_B, max_T
        self.cfg = config_of(shape)
        nbytes = workspace_bytes(shape, max_B, max_T, precision)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.stream = stream
        h = ctypes.c_void_p()
        check(lib.gpt2_build(ctypes.byref(self.cfg), max_B, max_T, PRECISIONS[precision],
                             self.workspace.data_ptr(), nbytes, _stream_handle(stream),
                             ctypes.byref(h)), "gpt2_build")
        self.handle = h
        nr, nf = ctypes.c_size_t(0), ctypes.c_size_t(0)
        check(lib.gpt2_num_parameters(h, ctypes.byref(nr), ctypes.byref(nf)), "gpt2_num_parameters")
        self.num_parameters, self.n_flat = nr.value, nf.value
        self.tensor_slices = {}
        for i, name in enumerate(PARAM_ORDER):
            off, n = ctypes.c_size_t(0), ctypes.c_size_t(0)
            check(lib.gpt2_param_tensor(h, i, ctypes.byref(off), ctypes.byref(n)), "gpt2_param_tensor")
            self.tensor_slices[name] = (off.value, n.value)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            lib.gpt2_free(h)
            self.handle = None

    # ---- views into the caller-owned workspace
    def _flat_view(self, ptr: int):
        import torch
        base = self.workspace.data_ptr()
        off = int(ptr) - base
        return self.workspace[off:off + self.n_flat * 4].view(torch.float32)

    def flat_params(self):
        return self._flat_view(lib.gpt2_params(self.handle))

    def flat_grads(self):
        return self._flat_view(lib.gpt2_grads(self.handle))

    def _split(self, flat):
        from step_gpt_train_03_b300.synth import param_shapes
        shapes = param_shapes(self.shape)
        return {k: flat[o:o + n].view(shapes[k]) for k, (o, n) in self.tensor_slices.items()}

    def params(self):
        return self._split(self.flat_params())

    def grads(self):
        return self._split(self.flat_grads())

    def load_params(self, params: dict) -> None:
        """Copy host arrays (name -> ndarray) into the fp32 master buffer, then sync."""
        import torch
        views = self.params()
        for name in PARAM_ORDER:
            views[name].copy_(torch.from_numpy(np.ascontiguousarray(params[name], np.float32)))
        self.sync_params()

    def adam_state(self):
        """(m, v) views of the AdamW moments, per tensor."""
        return (self._split(self._flat_view(lib.gpt2_adam_m(self.handle))),
                self._split(self._flat_view(lib.gpt2_adam_v(self.handle))))

    def load_state(self, params: dict, m: dict, v: dict) -> None:
        """Load master weights and both AdamW moments (name -> array each)."""
        import torch
        self.load_params(params)
        vm, vv = self.adam_state()
        for name in PARAM_ORDER:
            vm[name].copy_(torch.from_numpy(np.ascontiguousarray(m[name], np.float32)))
            vv[name].copy_(torch.from_numpy(np.ascontiguousarray(v[name], np.float32)))

    def sync_params(self):
        check(lib.gpt2_sync_params(self.handle), "gpt2_sync_params")

    def set_stream(self, stream):
        self.stream = stream
        check(lib.gpt2_set_stream(self.handle, _stream_handle(stream)), "gpt2_set_stream")

    # ---- the step
    def forward(self, tokens, targets=None, want_loss=True):
        """tokens/targets: int32 CUDA tensors (B, T).  Returns the mean loss (synchronises)
        when want_loss, else None (no synchronisation)."""
        B, T = tokens.shape
        self.last_B = B
        loss = ctypes.c_float(0.0)
        st = lib.gpt2_forward(self.handle, _ptr(tokens), _ptr(targets), B, T,
                              ctypes.byref(loss) if want_loss else None)
        check(st, "gpt2_forward")
        return loss.value if want_loss else None

    def zero_grad(self):
        check(lib.gpt2_zero_grad(self.handle), "gpt2_zero_grad")

    def backward(self):
        check(lib.gpt2_backward(self.handle), "gpt2_backward")

    def update(self, lr, beta1, beta2, eps, weight_decay, t):
        check(lib.gpt2_update(self.handle, lr, beta1, beta2, eps, weight_decay, t), "gpt2_update")

    def update_muon(self, lr_muon, momentum, ns_iters, lr, beta1, beta2, eps, weight_decay, t):
        check(lib.gpt2_update_muon(self.handle, lr_muon, momentum, ns_iters, lr, beta1, beta2, eps, weight_decay, t),
              "gpt2_update_muon")

    def step(self, tokens, targets, lr, beta1, beta2, eps, weight_decay, t, want_loss=True):
        loss = self.forward(tokens, targets, want_loss)
        self.zero_grad()
        self.backward()
        self.update(lr, beta1, beta2, eps, weight_decay, t)
        return loss

    def step_host(self, tokens_host, targets_host, lr, beta1, beta2, eps, weight_decay, t):
        """Whole step from host int32 buffers (torch CPU tensors, pinned for speed)."""
        B, T = tokens_host.shape
        loss = ctypes.c_float(0.0)
        check(lib.gpt2_step_host(self.handle, tokens_host.data_ptr(), targets_host.data_ptr(), B, T,
                                 lr, beta1, beta2, eps, weight_decay, t, ctypes.byref(loss)),
              "gpt2_step_host")
        return loss.value

    def step_device(self, tokens, targets, lr, beta1, beta2, eps, weight_decay, t, want_loss=False):
        """Whole step from int32 CUDA tensors (B, T) through gpt2_step (a CUDA graph once
        the shape has been seen).  Returns the mean loss (synchronises) when want_loss."""
        B, T = tokens.shape
        loss = ctypes.c_float(0.0)
        check(lib.gpt2_step(self.handle, _ptr(tokens), _ptr(targets), B, T, lr, beta1, beta2, eps,
                            weight_decay, t, ctypes.byref(loss) if want_loss else None), "gpt2_step")
        return loss.value if want_loss else None

    def step_muon_device(self, tokens, targets, lr_muon, momentum, ns_iters, lr, beta1, beta2, eps, weight_decay, t,
                         want_loss=False):
        """Whole Muon step from int32 CUDA tensors (B, T) through gpt2_step_muon (a CUDA graph
        once the shape has been seen).  Returns the mean loss (synchronises) when want_loss."""
        B, T = tokens.shape
        loss = ctypes.c_float(0.0)
        check(lib.gpt2_step_muon(self.handle, _ptr(tokens), _ptr(targets), B, T, lr_muon, momentum, ns_iters, lr,
                                 beta1, beta2, eps, weight_decay, t, ctypes.byref(loss) if want_loss else None),
              "gpt2_step_muon")
        return loss.value if want_loss else None

    def sample(self, pos: int, temperature: float, seed: int, out=None):
        """Next token of every sequence of the last forward (run without targets), from the
        logits at position `pos` (see gpt2_sample).  Returns an int32 CUDA tensor (B,)."""
        import torch
        B = self.last_B
        if out is None:
            out = torch.empty(B, dtype=torch.int32, device="cuda")
        check(lib.gpt2_sample(self.handle, pos, temperature, seed, _ptr(out)), "gpt2_sample")
        return out

    def generate(self, prompt, n_new: int, temperature: float, seed: int):
        """Extend int32 CUDA token sequences (B, T0) by n_new sampled tokens: one full
        forward of the sequence so far per new token, sampled at its last position (the
        sampler's seed advances by B per token).  Returns (B, T0 + n_new)."""
        import torch
        toks = prompt.clone()
        for i in range(n_new):
            self.forward(toks, None, want_loss=False)
            nxt = self.sample(toks.shape[1] - 1, temperature, seed + i * toks.shape[0])
            toks = torch.cat([toks, nxt.view(-1, 1)], dim=1).contiguous()
        return toks

    def save(self, path: str):
        """Write the fp32 master weights to a parameter file (see gpt2_save_params)."""
        check(lib.gpt2_save_params(self.handle, str(path).encode()), "gpt2_save_params")

    def load(self, path: str):
        """Load a parameter file written for this configuration (see gpt2_load_params)."""
        check(lib.gpt2_load_params(self.handle, str(path).encode()), "gpt2_load_params")

    def set_graphs(self, enable: bool):
        check(lib.gpt2_set_graphs(self.handle, 1 if enable else 0), "gpt2_set_graphs")

    def losses(self, n):
        import torch
        ptr = lib.gpt2_losses(self.handle)
        off = int(ptr) - self.workspace.data_ptr()
        return self.workspace[off:off + n * 4].view(torch.float32)

    def loss_device(self):
        import torch
        ptr = lib.gpt2_loss(self.handle)
        off = int(ptr) - self.workspace.data_ptr()
        return self.workspace[off:off + 4].view(torch.float32)

    def check(self):
        check(lib.gpt2_check(self.handle), "gpt2_check")

    def fp8_weights(self, which: str):
        """(codes uint8 (L, rows, C), deq fp32 (L,)) views of the fp8 mode's weight shadow of
        'qkvw' or 'fcw'."""
        import torch
        codes, deq = ctypes.c_void_p(), ctypes.c_void_p()
        check(lib.gpt2_fp8_weights(self.handle, 0 if which == "qkvw" else 1, ctypes.byref(codes), ctypes.byref(deq)),
              "gpt2_fp8_weights")
        L, C = self.shape.num_layers, self.shape.channels
        rows = 3 * C if which == "qkvw" else 4 * C
        base = self.workspace.data_ptr()
        c_off, d_off = codes.value - base, deq.value - base
        return (self.workspace[c_off:c_off + L * rows * C].view(L, rows, C),
                self.workspace[d_off:d_off + 4 * L].view(torch.float32))


# ---- observability -----------------------------------------------------------------------------
def kernel_launches() -> int:
    return int(lib.gpt2_kernel_launches())


def profile_classes() -> list:
    return [lib.gpt2_profile_class_name(c).decode() for c in range(lib.gpt2_profile_num_classes())]


def profile_enable(classes=None):
    """Trace the named kernel classes (all when None; [] switches tracing off)."""
    names = profile_classes()
    if classes is None:
        mask = (1 << len(names)) - 1
    else:
        mask = 0
        for c in classes:
            mask |= 1 << names.index(c)
    check(lib.gpt2_profile_enable(mask), "gpt2_profile_enable")


def profile_reset():
    check(lib.gpt2_profile_reset(), "gpt2_profile_reset")


def profile_read() -> dict:
    """Collect pending events; {class name: dict(ms, launches, flops, bytes)}."""
    check(lib.gpt2_profile_collect(), "gpt2_profile_collect")
    out = {}
    for c in range(lib.gpt2_profile_num_classes()):
        ms, n = ctypes.c_double(0), ctypes.c_longlong(0)
        fl, by = ctypes.c_double(0), ctypes.c_double(0)
        check(lib.gpt2_profile_read(c, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(fl),
                                    ctypes.byref(by)), "gpt2_profile_read")
        out[lib.gpt2_profile_class_name(c).decode()] = dict(ms=ms.value, launches=n.value,
                                                             flops=fl.value, bytes=by.value)
    return out


# ---- single-layer entry points -----------------------------------------------------------------
def layernorm_forward(out, mean, rstd, inp, weight, bias, stream=None):
    N, C = inp.shape
    check(lib.gpt2_layernorm_forward(_ptr(out), _ptr(mean), _ptr(rstd), _ptr(inp), _ptr(weight),
                                     _ptr(bias), N, C, _stream_handle(stream)), "gpt2_layernorm_forward")


def layernorm_backward_scratch_bytes(N, C) -> int:
    return int(lib.gpt2_layernorm_backward_scratch_bytes(N, C))


def layernorm_backward(dinp, dweight, dbias, dout, inp, weight, mean, rstd, scratch, stream=None):
    N, C = inp.shape
    check(lib.gpt2_layernorm_backward(_ptr(dinp), _ptr(dweight), _ptr(dbias), _ptr(dout), _ptr(inp),
                                      _ptr(weight), _ptr(mean), _ptr(rstd), N, C, _ptr(scratch),
                                      scratch.numel() * scratch.element_size(), _stream_handle(stream)),
          "gpt2_layernorm_backward")


NOALLOC_SCRATCH_BYTES = 4 << 20


def layernorm_backward_noalloc(dinp, dweight, dbias, dout, inp, weight, mean, rstd, stream=None):
    """gpt2_layernorm_backward_noalloc: the library's built-in scratch, no allocation."""
    N, C = inp.shape
    check(lib.gpt2_layernorm_backward_noalloc(_ptr(dinp), _ptr(dweight), _ptr(dbias), _ptr(dout),
                                              _ptr(inp), _ptr(weight), _ptr(mean), _ptr(rstd), N, C,
                                              _stream_handle(stream)), "gpt2_layernorm_backward_noalloc")


def attention_forward(out, lse, qkv, NH, precision, stream=None):
    """qkv (B,T,3C) -> out (B,T,C); lse (B,NH,T) fp32 (bf16) or probabilities (B,NH,T,T) (fp32)."""
    B, T, C3 = qkv.shape
    check(lib.gpt2_attention_forward(_ptr(out), _ptr(lse), _ptr(qkv), B, T, C3 // 3, NH, PRECISIONS[precision],
                                     _stream_handle(stream)), "gpt2_attention_forward")


def attention_backward_scratch_bytes(B, T, C, NH, precision) -> int:
    return int(lib.gpt2_attention_backward_scratch_bytes(B, T, C, NH, PRECISIONS[precision]))


def attention_backward(dqkv, dout, qkv, out, lse, NH, precision, scratch, dbias=None, stream=None):
    """gpt2_attention_backward: dqkv from dout; dbias (fp32 (3C), optional) += column sums of dqkv."""
    B, T, C3 = qkv.shape
    check(lib.gpt2_attention_backward(_ptr(dqkv), _ptr(dbias), _ptr(dout), _ptr(qkv), _ptr(out), _ptr(lse), B, T,
                                      C3 // 3, NH, PRECISIONS[precision], _ptr(scratch),
                                      scratch.numel() * scratch.element_size(), _stream_handle(stream)),
          "gpt2_attention_backward")


def matmul_forward(out, inp, weight, bias, precision, stream=None):
    M, K = inp.shape
    N = weight.shape[0]
    check(lib.gpt2_matmul_forward(_ptr(out), _ptr(inp), _ptr(weight), _ptr(bias), M, N, K,
                                  PRECISIONS[precision], _stream_handle(stream)), "gpt2_matmul_forward")


EPILOGUES = {"bias": 0, "gelu": 1, "residual": 2}


def matmul_forward_fused(out, aux, inp, weight, bias, epilogue, precision, stream=None):
    """gpt2_matmul_forward_fused: out = epilogue(inp weight^T + bias); aux is the GELU
    pre-activation (written) or the residual input (read)."""
    M, K = inp.shape
    N = weight.shape[0]
    check(lib.gpt2_matmul_forward_fused(_ptr(out), _ptr(aux), _ptr(inp), _ptr(weight), _ptr(bias), M, N, K,
                                        EPILOGUES[epilogue], PRECISIONS[precision], _stream_handle(stream)),
          "gpt2_matmul_forward_fused")


def matmul_backward_input_gelu_scratch_bytes(M, K) -> int:
    return int(lib.gpt2_matmul_backward_input_gelu_scratch_bytes(M, K))


def matmul_backward_input_gelu(dinp, dout, weight, pre, precision, dbias=None, scratch=None, stream=None):
    """gpt2_matmul_backward_input_gelu: dinp = (dout weight) * gelu'(pre); dbias (fp32 (K),
    optional, with scratch) += column sums of dinp."""
    M, N = dout.shape
    K = weight.shape[1]
    nbytes = scratch.numel() * scratch.element_size() if scratch is not None else 0
    check(lib.gpt2_matmul_backward_input_gelu(_ptr(dinp), _ptr(dbias), _ptr(dout), _ptr(weight), _ptr(pre), M, N, K,
                                              PRECISIONS[precision], _ptr(scratch), nbytes, _stream_handle(stream)),
          "gpt2_matmul_backward_input_gelu")


def layernorm_forward_fp8(out, codes, row_deq, mean, rstd, inp, weight, bias, stream=None):
    """gpt2_layernorm_forward_fp8 (fp32 tensors, codes uint8 (N, C), row_deq fp32 (N))."""
    N, C = inp.shape
    check(lib.gpt2_layernorm_forward_fp8(_ptr(out), _ptr(codes), _ptr(row_deq), _ptr(mean), _ptr(rstd), _ptr(inp),
                                         _ptr(weight), _ptr(bias), N, C, _stream_handle(stream)),
          "gpt2_layernorm_forward_fp8")


def quantize_e4m3(codes, deq, amax_scratch, x, stream=None):
    """gpt2_quantize_e4m3: per-tensor e4m3 codes of the fp32 tensor x."""
    check(lib.gpt2_quantize_e4m3(_ptr(codes), _ptr(deq), _ptr(amax_scratch), _ptr(x), x.numel(),
                                 _stream_handle(stream)), "gpt2_quantize_e4m3")


def matmul_forward_fp8(out, aux, inp, inp_deq, weight, weight_deq, bias, epilogue, stream=None):
    """gpt2_matmul_forward_fp8: inp (M,K) and weight (N,K) e4m3 codes (uint8 tensors)."""
    M, K = inp.shape
    N = weight.shape[0]
    check(lib.gpt2_matmul_forward_fp8(_ptr(out), _ptr(aux), _ptr(inp), _ptr(inp_deq), _ptr(weight),
                                      _ptr(weight_deq), _ptr(bias), M, N, K, EPILOGUES[epilogue],
                                      _stream_handle(stream)), "gpt2_matmul_forward_fp8")


def newton_schulz(out, G, iters, stream=None):
    """gpt2_newton_schulz: out (r, c) bf16 = iters Newton-Schulz steps from G (r, c) fp32."""
    import torch
    r, c = G.shape
    nb = int(lib.gpt2_newton_schulz_scratch_bytes(r, c))
    sc = torch.empty(nb, dtype=torch.uint8, device=G.device)
    check(lib.gpt2_newton_schulz(_ptr(out), _ptr(G), r, c, iters, _ptr(sc), nb, _stream_handle(stream)),
          "gpt2_newton_schulz")


def layer_check(stream=None):
    """gpt2_layer_check: synchronise and raise if a single-layer kernel's bounded wait ran out."""
    check(lib.gpt2_layer_check(_stream_handle(stream)), "gpt2_layer_check")


def matmul_backward_scratch_bytes(M, N) -> int:
    return int(lib.gpt2_matmul_backward_scratch_bytes(M, N))


def matmul_backward(dinp, dweight, dbias, dout, inp, weight, precision, scratch, stream=None):
    M, K = inp.shape
    N = weight.shape[0]
    check(lib.gpt2_matmul_backward(_ptr(dinp), _ptr(dweight), _ptr(dbias), _ptr(dout), _ptr(inp),
                                   _ptr(weight), M, N, K, PRECISIONS[precision], _ptr(scratch),
                                   scratch.numel() * scratch.element_size(), _stream_handle(stream)),
          "gpt2_matmul_backward")
