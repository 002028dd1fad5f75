"""ctypes binding of libgpt2 (include/gpt2.h, include/gpt2_ops.h).

Argument marshalling only: every step of the training step runs in the library's CUDA
kernels. Device buffers may be given as torch CUDA tensors or raw integer addresses;
streams as torch.cuda.Stream or raw cudaStream_t integers. The library must have been
built (decoder_only_transformer_05_b300.build); loading fails loudly otherwise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgpt2.so")

GPT2_OK = 0
ERRORS = {-1: "INVALID_CONFIG", -2: "OOM", -3: "CUDA", -4: "BAD_TOKEN", -5: "SEQ_TOO_LONG",
          -6: "TIMEOUT", -7: "STATE", -8: "ARG"}
FP32, BF16 = 0, 1
REGION = dict(params=0, grads=1, m=2, v=3, params_bf16=4, logits=5, losses=6, encoded=7,
              argmax=8)
EPI = dict(store=0, gelu_fwd=1, gelu_bwd=2, accum=3, gelu_fwd_u=4, gelu_bwd_u=5, logits_ce=6)
PROF = dict(gemm=0, attention=1, layernorm=2, classifier=3, encoder=4, optimizer=5, other=6)


class GPT2Error(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code
        self.name = ERRORS.get(code, str(code))


class _Config(ctypes.Structure):
    _fields_ = [("vocab_size", ctypes.c_int32), ("padded_vocab_size", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("n_layer", ctypes.c_int32),
                ("n_head", ctypes.c_int32), ("n_embd", ctypes.c_int32),
                ("bias", ctypes.c_int32), ("precision", ctypes.c_int32),
                ("batch_size", ctypes.c_int32), ("init", ctypes.c_int32),
                ("seed", ctypes.c_uint64), ("recompute", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> (restype, argtypes): the complete exported interface of the two headers
SIGNATURES = {
    "gpt2_create": (_I, [ctypes.POINTER(_Config), ctypes.POINTER(_P)]),
    "gpt2_host_init": (_I, [ctypes.POINTER(_Config), _P, _SZ]),
    "gpt2_host_num_params": (_I, [ctypes.POINTER(_Config), ctypes.POINTER(_SZ),
                                  ctypes.POINTER(_SZ)]),
    "gpt2_set_stream": (_I, [_P, _P]),
    "gpt2_forward": (_I, [_P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_F)]),
    "gpt2_backward": (_I, [_P, _F]),
    "gpt2_zero_grad": (_I, [_P]),
    "gpt2_forward_backward": (_I, [_P, _P, _P, ctypes.c_int32, ctypes.c_int32, _F]),
    "gpt2_set_graph_mode": (_I, [_P, _I]),
    "gpt2_prefill": (_I, [_P, _P, ctypes.c_int32, ctypes.c_int32, _P]),
    "gpt2_decode_step": (_I, [_P, _P, ctypes.c_int32, _P]),
    "gpt2_decode_length": (_I, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "gpt2_adamw_step": (_I, [_P, _F, _F, _F, _F, _F, _F, ctypes.POINTER(_F)]),
    "gpt2_get_loss": (_I, [_P, ctypes.POINTER(_F)]),
    "gpt2_sync": (_I, [_P]),
    "gpt2_num_tensors": (_I, [_P]),
    "gpt2_tensor_info": (_I, [_P, _I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_SZ),
                              ctypes.POINTER(_I), ctypes.POINTER(_I64)]),
    "gpt2_num_params": (_I, [_P, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "gpt2_copy_region": (_I, [_P, _I, _SZ, _P, _SZ, _I]),
    "gpt2_region_ptr": (_I, [_P, _I, ctypes.POINTER(_P), ctypes.POINTER(_SZ)]),
    "gpt2_get_step": (_I, [_P, ctypes.POINTER(_I64)]),
    "gpt2_set_step": (_I, [_P, _I64]),
    "gpt2_profile_enable": (_I, [_P, _I, _I]),
    "gpt2_profile_read": (_I, [_P, _I, ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_double), _I]),
    "gpt2_memory_bytes": (_I, [_P, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "gpt2_last_error": (ctypes.c_char_p, []),
    "gpt2_kernel_launches": (_I64, []),
    "gpt2_destroy": (None, [_P]),
    "gpt2_op_gemm": (_I, [_I, _I, _I, _I, _P, _I64, _I, _P, _I64, _I, _I, _P, _I64, _P, _P, _P,
                          _P, _P, _F, _I, _P, _SZ, _P]),
    "gpt2_op_attention_forward": (_I, [_I, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gpt2_op_attention_backward": (_I, [_I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gpt2_op_layernorm_forward": (_I, [_I, _P, _P, _P, _P, _P, _P, _I, _I, _P]),
    "gpt2_op_layernorm_partials_floats": (_SZ, [_I, _I]),
    "gpt2_op_layernorm_backward": (_I, [_I, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _F,
                                        _P, _P]),
    "gpt2_op_classifier": (_I, [_I, _P, _P, _P, _I, _I, _I, _P, _P]),
    "gpt2_op_layernorm_backward_noalloc": (_I, [_I, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I,
                                                _I, _F, _P]),
    "gpt2_debug_gemm_waits": (_I, [_I64, _I]),
    "gpt2_op_lmhead_ce_scratch_bytes": (_SZ, [_I, _I]),
    "gpt2_op_lmhead_cross_entropy": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
}

_lib = None


def load_library(path: str = LIB_PATH):
    """Load libgpt2.so and declare every entry point; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libgpt2.so not built at {path}; run "
                          "python -m decoder_only_transformer_05_b300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def kernel_launches():
    """Kernels the library has launched in this process."""
    return load_library().gpt2_kernel_launches()


def _check(rc):
    if rc != GPT2_OK:
        msg = _lib.gpt2_last_error()
        raise GPT2Error(rc, msg.decode() if msg else "")


def ptr(x):
    """Device address of a torch tensor, or the integer itself (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def stream_handle(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def make_config(vocab_size, block_size, n_layer, n_head, n_embd, batch_size,
                padded_vocab_size=0, bias=True, precision="bf16", init=True, seed=0,
                recompute=False):
    return _Config(vocab_size, padded_vocab_size, block_size, n_layer, n_head, n_embd,
                   int(bool(bias)), BF16 if precision == "bf16" else FP32, batch_size,
                   int(bool(init)), seed & 0xFFFFFFFFFFFFFFFF, int(bool(recompute)))


def host_num_params(**cfg):
    """(model parameter count, flat buffer elements) for a config, without a GPU."""
    lib = load_library()
    c = make_config(**cfg)
    a, b = _SZ(), _SZ()
    _check(lib.gpt2_host_num_params(ctypes.byref(c), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def host_init(**cfg):
    """The flat initial parameter buffer (float32) gpt2_create uploads, without a GPU."""
    lib = load_library()
    c = make_config(**cfg)
    _, n = host_num_params(**cfg)
    out = np.empty(n, dtype=np.float32)
    _check(lib.gpt2_host_init(ctypes.byref(c), out.ctypes.data, n))
    return out


class GPT2:
    """One model instance on the current CUDA device (see include/gpt2.h)."""

    def __init__(self, vocab_size, block_size, n_layer, n_head, n_embd, batch_size,
                 padded_vocab_size=0, bias=True, precision="bf16", init=True, seed=0,
                 recompute=False):
        lib = load_library()
        cfg = make_config(vocab_size, block_size, n_layer, n_head, n_embd, batch_size,
                          padded_vocab_size, bias, precision, init, seed, recompute)
        h = _P()
        _check(lib.gpt2_create(ctypes.byref(cfg), ctypes.byref(h)))
        self._h = h
        self.lib = lib
        self.precision = precision
        self.C, self.V = n_embd, vocab_size
        n_model, n_buf = _SZ(), _SZ()
        _check(lib.gpt2_num_params(h, ctypes.byref(n_model), ctypes.byref(n_buf)))
        self.num_params, self.buffer_elems = n_model.value, n_buf.value
        self.Vp = self.tensor_table()["wte"][1][0]

    # ------------------------------------------------------------------ lifecycle
    def close(self):
        if getattr(self, "_h", None):
            self.lib.gpt2_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def memory_bytes(self):
        """(parameter block bytes, all other device bytes) the handle holds."""
        a, b = _SZ(), _SZ()
        _check(self.lib.gpt2_memory_bytes(self._h, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def set_stream(self, stream):
        _check(self.lib.gpt2_set_stream(self._h, stream_handle(stream)))

    # ------------------------------------------------------------------ the step
    def forward(self, tokens, targets=None, B=None, T=None, want_loss=False):
        if B is None:
            B, T = tokens.shape
        loss = _F()
        _check(self.lib.gpt2_forward(self._h, ptr(tokens), ptr(targets), B, T,
                                     ctypes.byref(loss) if want_loss else None))
        return loss.value if want_loss else None

    def backward(self, loss_scale=1.0):
        _check(self.lib.gpt2_backward(self._h, loss_scale))

    def forward_backward(self, tokens, targets, B=None, T=None, loss_scale=1.0):
        """forward(tokens, targets) then backward(loss_scale); tokens and targets may live on
        the device or in (pinned) host memory. Replayed as a CUDA graph after the first call
        of each shape unless set_graph_mode(False)."""
        if B is None:
            B, T = tokens.shape
        _check(self.lib.gpt2_forward_backward(self._h, ptr(tokens), ptr(targets), B, T,
                                              loss_scale))

    # ------------------------------------------------------------------ inference
    def prefill(self, tokens, next_tokens, B=None, T0=None):
        """Forward over the prompt [B, T0] with the key/value cache filled; the argmax token of
        each row's last position goes to next_tokens [B] (device int32)."""
        if B is None:
            B, T0 = tokens.shape
        _check(self.lib.gpt2_prefill(self._h, ptr(tokens), B, T0, ptr(next_tokens)))

    def decode_step(self, tokens, next_tokens, B=None):
        """One new token per row (tokens [B] device int32) through the cached model; its
        logits' argmax goes to next_tokens [B]."""
        if B is None:
            B = tokens.shape[0]
        _check(self.lib.gpt2_decode_step(self._h, ptr(tokens), B, ptr(next_tokens)))

    @property
    def decode_length(self):
        n = ctypes.c_int32()
        _check(self.lib.gpt2_decode_length(self._h, ctypes.byref(n)))
        return n.value

    def generate(self, prompt, n_new):
        """Greedy decoding: prompt [B, T0] (device int32) -> the n_new tokens [B, n_new] chosen
        by argmax, each fed back as the next input."""
        import torch
        B = prompt.shape[0]
        out = torch.empty(B, n_new, dtype=torch.int32, device=prompt.device)
        nxt = torch.empty(B, dtype=torch.int32, device=prompt.device)
        self.prefill(prompt, nxt)
        for i in range(n_new):
            out[:, i] = nxt
            if i + 1 < n_new:
                self.decode_step(out[:, i].contiguous(), nxt)
        return out

    def set_graph_mode(self, enabled):
        _check(self.lib.gpt2_set_graph_mode(self._h, int(bool(enabled))))

    def zero_grad(self):
        _check(self.lib.gpt2_zero_grad(self._h))

    def adamw_step(self, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, grad_clip=0.0,
                   want_norm=False):
        n = _F()
        _check(self.lib.gpt2_adamw_step(self._h, lr, beta1, beta2, eps, weight_decay, grad_clip,
                                        ctypes.byref(n) if want_norm else None))
        return n.value if want_norm else None

    def get_loss(self):
        v = _F()
        _check(self.lib.gpt2_get_loss(self._h, ctypes.byref(v)))
        return v.value

    def sync(self):
        _check(self.lib.gpt2_sync(self._h))

    @property
    def step(self):
        t = _I64()
        _check(self.lib.gpt2_get_step(self._h, ctypes.byref(t)))
        return t.value

    @step.setter
    def step(self, t):
        _check(self.lib.gpt2_set_step(self._h, t))

    # ------------------------------------------------------------------ memory
    def tensor_table(self):
        """name -> (element offset, shape)"""
        out = {}
        for i in range(self.lib.gpt2_num_tensors(self._h)):
            name, off, nd = ctypes.c_char_p(), _SZ(), _I()
            shape = (_I64 * 3)()
            _check(self.lib.gpt2_tensor_info(self._h, i, ctypes.byref(name), ctypes.byref(off),
                                             ctypes.byref(nd), shape))
            out[name.value.decode()] = (off.value, tuple(shape[:nd.value]))
        return out

    def region_ptr(self, region):
        p, n = _P(), _SZ()
        _check(self.lib.gpt2_region_ptr(self._h, REGION[region], ctypes.byref(p),
                                        ctypes.byref(n)))
        return p.value, n.value

    def read_region(self, region, dtype, count=None, offset_elems=0):
        dt = np.dtype(dtype)
        _, nbytes = self.region_ptr(region)
        if count is None:
            count = nbytes // dt.itemsize - offset_elems
        out = np.empty(count, dtype=dt)
        _check(self.lib.gpt2_copy_region(self._h, REGION[region], offset_elems * dt.itemsize,
                                         out.ctypes.data, out.nbytes, 0))
        return out

    def write_region(self, region, array, offset_elems=0):
        a = np.ascontiguousarray(array)
        _check(self.lib.gpt2_copy_region(self._h, REGION[region], offset_elems * a.itemsize,
                                         a.ctypes.data, a.nbytes, 1))

    def _unflatten(self, flat):
        return {name: flat[off:off + int(np.prod(shape))].reshape(shape).copy()
                for name, (off, shape) in self.tensor_table().items()}

    def get_params(self):
        return self._unflatten(self.read_region("params", np.float32))

    def get_grads(self):
        return self._unflatten(self.read_region("grads", np.float32))

    def get_moments(self):
        return (self._unflatten(self.read_region("m", np.float32)),
                self._unflatten(self.read_region("v", np.float32)))

    def set_params(self, params: dict, region="params"):
        flat = self.read_region(region, np.float32)
        for name, (off, shape) in self.tensor_table().items():
            flat[off:off + int(np.prod(shape))] = np.asarray(params[name], np.float32).reshape(-1)
        self.write_region(region, flat)

    # ------------------------------------------------------------------ profiling
    def profile_enable(self, classes=("gemm",), capacity=65536):
        mask = 0
        for c in classes:
            mask |= 1 << PROF[c]
        _check(self.lib.gpt2_profile_enable(self._h, mask, capacity))

    def profile_read(self, cls, reset=False):
        n, ms, work = _I64(), ctypes.c_double(), ctypes.c_double()
        _check(self.lib.gpt2_profile_read(self._h, PROF[cls], ctypes.byref(n), ctypes.byref(ms),
                                          ctypes.byref(work), int(reset)))
        return n.value, ms.value, work.value


# ---------------------------------------------------------------------- single ops
def _prec(p):
    return BF16 if p in ("bf16", BF16) else FP32


def op_gemm(precision, M, N, K, A, lda, a_mn, B, ldb, b_mn, epi="store", out=None, ldo=None,
            bias=None, resid=None, pre=None, aux=None, accum=None, scale=1.0, splits=1,
            workspace=None, workspace_bytes=0, stream=None):
    lib = load_library()
    _check(lib.gpt2_op_gemm(_prec(precision), M, N, K, ptr(A), lda, int(a_mn), ptr(B), ldb,
                            int(b_mn), EPI[epi], ptr(out), ldo if ldo is not None else N,
                            ptr(bias), ptr(resid), ptr(pre), ptr(aux), ptr(accum), scale, splits,
                            ptr(workspace), workspace_bytes, stream_handle(stream)))


def op_attention_forward(precision, out, lse, qkv, B, T, C, H, stream=None):
    lib = load_library()
    _check(lib.gpt2_op_attention_forward(_prec(precision), ptr(out), ptr(lse), ptr(qkv), B, T, C,
                                         H, stream_handle(stream)))


def op_attention_backward(precision, dqkv, Dbuf, dout, out, qkv, lse, B, T, C, H, stream=None):
    lib = load_library()
    _check(lib.gpt2_op_attention_backward(_prec(precision), ptr(dqkv), ptr(Dbuf), ptr(dout),
                                          ptr(out), ptr(qkv), ptr(lse), B, T, C, H,
                                          stream_handle(stream)))


def op_layernorm_forward(precision, y, mean, rstd, x, w, b, M, C, stream=None):
    lib = load_library()
    _check(lib.gpt2_op_layernorm_forward(_prec(precision), ptr(y), ptr(mean), ptr(rstd), ptr(x),
                                         ptr(w), ptr(b), M, C, stream_handle(stream)))


def op_layernorm_partials_floats(M, C):
    return load_library().gpt2_op_layernorm_partials_floats(M, C)


def op_layernorm_backward(precision, dres, accumulate, dw, db, dy, x, w, mean, rstd, M, C,
                          scale, partials, stream=None):
    lib = load_library()
    _check(lib.gpt2_op_layernorm_backward(_prec(precision), ptr(dres), int(accumulate), ptr(dw),
                                          ptr(db), ptr(dy), ptr(x), ptr(w), ptr(mean), ptr(rstd),
                                          M, C, scale, ptr(partials), stream_handle(stream)))


def op_classifier(precision, logits, losses, targets, M, V, Vp, err, stream=None):
    lib = load_library()
    _check(lib.gpt2_op_classifier(_prec(precision), ptr(logits), ptr(losses), ptr(targets), M, V,
                                  Vp, ptr(err), stream_handle(stream)))


def op_layernorm_backward_noalloc(precision, dres, accumulate, dw, db, dy, x, w, mean, rstd, M,
                                  C, scale, stream=None):
    """LayerNorm backward with the library's built-in scratch (no partials buffer)."""
    lib = load_library()
    _check(lib.gpt2_op_layernorm_backward_noalloc(_prec(precision), ptr(dres), int(accumulate),
                                                  ptr(dw), ptr(db), ptr(dy), ptr(x), ptr(w),
                                                  ptr(mean), ptr(rstd), M, C, scale,
                                                  stream_handle(stream)))


def debug_gemm_waits(wait_limit_ns=0, drop_first_signal=False):
    """Test hook of the GEMM's bounded waits (see include/gpt2_ops.h); (0, False) = off."""
    lib = load_library()
    _check(lib.gpt2_debug_gemm_waits(int(wait_limit_ns), int(bool(drop_first_signal))))


def op_lmhead_ce_scratch_bytes(M, Vp):
    return load_library().gpt2_op_lmhead_ce_scratch_bytes(M, Vp)


def op_lmhead_cross_entropy(M, C, V, Vp, x, wte, targets, logits, losses, scratch, err,
                            stream=None):
    """bf16 lm_head GEMM with the cross-entropy's softmax statistics in its epilogue, then
    the losses and the dlogits (in place over the logits) in one pass."""
    lib = load_library()
    _check(lib.gpt2_op_lmhead_cross_entropy(M, C, V, Vp, ptr(x), ptr(wte), ptr(targets),
                                            ptr(logits), ptr(losses), ptr(scratch),
                                            scratch.numel() * scratch.element_size(), ptr(err),
                                            stream_handle(stream)))
