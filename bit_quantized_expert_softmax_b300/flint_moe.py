"""ctypes binding of libflint_moe.so (the C ABI declared in include/flint_moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Functions keep the C names; device buffers are torch CUDA tensors
(PyTorch supplies device memory and streams). There is no CPU fallback: if the
library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libflint_moe.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "flint_moe.h")

FLINT_OK, FLINT_EINVAL, FLINT_ENOMEM, FLINT_ECUDA, FLINT_ESTATE, FLINT_ETIMEOUT, \
    FLINT_ENOTIMPL, FLINT_EDEVICE = range(8)
FLINT_W_NVFP4, FLINT_W_Q4_1 = 0, 1


class flint_moe_config(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("f", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("n_shared", ctypes.c_int), ("wfmt", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("n_layers", ctypes.c_int), ("device", ctypes.c_int)]


class flint_moe_attn_config(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int), ("n_kv", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("window", ctypes.c_int), ("cap", ctypes.c_int), ("rope", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("eps", ctypes.c_float)]


class flint_moe_weights(ctypes.Structure):
    _fields_ = [("router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p)]


class FlintError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m bit_quantized_expert_softmax_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "flint_moe_create": (_I, [ctypes.POINTER(flint_moe_config), ctypes.POINTER(_P)]),
            "flint_moe_load_weights": (_I, [_P, _I, ctypes.POINTER(flint_moe_weights)]),
            "flint_moe_forward": (_I, [_P, _I, _P, _I, _P, _P]),
            "flint_moe_forward_stack": (_I, [_P, _I, _I, _P, _I, _P]),
            "flint_moe_destroy": (None, [_P]),
            "flint_moe_status": (_I, [_P]),
            "flint_moe_status_string": (ctypes.c_char_p, [_I]),
            "flint_moe_router": (_I, [_P, _I, _P, _I, _P, _P, _P, _P]),
            "flint_moe_topk": (_I, [_P, _I, _I, _I, _P, _P, _P]),
            "flint_moe_bucket": (_I, [_P, _P, _I, _P, _P, _P]),
            "flint_moe_dequant": (_I, [_P, _I, _I, _I, _P, _P]),
            "flint_moe_device_bytes": (ctypes.c_size_t, [_P]),
            "flint_moe_launch_count": (ctypes.c_uint64, [_P]),
            "flint_moe_forward_launches": (_I, [_P, _I]),
            "flint_moe_tensor_core_plan": (_I, [_P, _I, _I]),
            "flint_moe_debug_fp4_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
            "flint_moe_debug_act_quant": (_I, [_P, _I, _I, _P, _P, _P, _P]),
            "flint_moe_profile_begin": (_I, [_P, _I]),
            "flint_moe_profile_end": (_I, [_P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(_I)]),
            "flint_moe_load_lm_head": (_I, [_P, _I, _P, _P, ctypes.c_float]),
            "flint_moe_lm_head": (_I, [_P, _P, _I, _P, _P]),
            "flint_moe_sample": (_I, [_P, _P, _I, ctypes.c_float, _I, ctypes.c_float, _P, _P, _P, _P]),
            "flint_moe_probe_fp4_peak": (_I, [_I, _I, ctypes.POINTER(ctypes.c_float),
                                              ctypes.POINTER(ctypes.c_double)]),
            "flint_moe_debug_wait_timeout": (_I, [_P, _I, ctypes.c_uint32, _P]),
            "flint_moe_quantize_nvfp4": (_I, [_P, _I, _I, _P, _P, _P, _P]),
            "flint_moe_attn_decode": (_I, [ctypes.POINTER(flint_moe_attn_config), _I, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/flint_moe.h declares."""
    with open(HEADER_PATH) as fh:
        text = fh.read()
    return re.findall(r"FLINT_API\s+[\w\s\*]+?\b(flint_moe_\w+)\s*\(", text)


def status_string(code: int) -> str:
    try:
        return lib().flint_moe_status_string(int(code)).decode()
    except Exception:   # library missing: still give a readable message
        return f"status {code}"


def _check(code: int, what: str) -> None:
    if code != FLINT_OK:
        raise FlintError(code, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------------------
# thin wrappers with the C names
# ---------------------------------------------------------------------------


def flint_moe_create(d: int, f: int, n_experts: int = 256, top_k: int = 6, n_shared: int = 1,
                     wfmt: int = FLINT_W_NVFP4, max_tokens: int = 64, n_layers: int = 1,
                     device: int = 0) -> int:
    cfg = flint_moe_config(d, f, n_experts, top_k, n_shared, wfmt, max_tokens, n_layers, device)
    h = _P()
    _check(lib().flint_moe_create(ctypes.byref(cfg), ctypes.byref(h)), "flint_moe_create")
    return h.value


def flint_moe_load_weights(h: int, layer: int, router: np.ndarray, router_bias, codes: np.ndarray,
                           scales: np.ndarray, tensor_scale) -> None:
    """Host numpy arrays in the canonical layout (see include/flint_moe.h)."""
    arrs = [np.ascontiguousarray(router, dtype=np.float32),
            None if router_bias is None else np.ascontiguousarray(router_bias, dtype=np.float32),
            np.ascontiguousarray(codes, dtype=np.uint8),
            np.ascontiguousarray(scales, dtype=np.uint8),
            None if tensor_scale is None else np.ascontiguousarray(tensor_scale, dtype=np.float32)]
    ptrs = [None if a is None else a.ctypes.data for a in arrs]
    w = flint_moe_weights(*ptrs)
    _check(lib().flint_moe_load_weights(h, layer, ctypes.byref(w)), "flint_moe_load_weights")


def flint_moe_forward(h: int, layer: int, hidden, T: int, out, stream=None) -> None:
    _check(lib().flint_moe_forward(h, layer, _ptr(hidden), T, _ptr(out), _stream(stream)),
           "flint_moe_forward")


def flint_moe_forward_stack(h: int, layer0: int, n_layers: int, hidden, T: int, stream=None) -> None:
    _check(lib().flint_moe_forward_stack(h, layer0, n_layers, _ptr(hidden), T, _stream(stream)),
           "flint_moe_forward_stack")


def flint_moe_destroy(h: int) -> None:
    lib().flint_moe_destroy(h)


def flint_moe_status(h: int) -> int:
    return int(lib().flint_moe_status(h))


def flint_moe_router(h: int, layer: int, hidden, T: int, logits=None, idx=None, w=None, stream=None) -> None:
    _check(lib().flint_moe_router(h, layer, _ptr(hidden), T, _ptr(logits), _ptr(idx), _ptr(w),
                                  _stream(stream)), "flint_moe_router")


def flint_moe_topk(logits, T: int, E: int, k: int, idx, w=None, stream=None) -> None:
    _check(lib().flint_moe_topk(_ptr(logits), T, E, k, _ptr(idx), _ptr(w), _stream(stream)),
           "flint_moe_topk")


def flint_moe_bucket(h: int, idx, T: int, offsets, perm, stream=None) -> None:
    _check(lib().flint_moe_bucket(h, _ptr(idx), T, _ptr(offsets), _ptr(perm), _stream(stream)),
           "flint_moe_bucket")


def flint_moe_dequant(h: int, layer: int, expert: int, mat: int, out, stream=None) -> None:
    _check(lib().flint_moe_dequant(h, layer, expert, mat, _ptr(out), _stream(stream)),
           "flint_moe_dequant")


def flint_moe_device_bytes(h: int) -> int:
    return int(lib().flint_moe_device_bytes(h))


def flint_moe_launch_count(h: int) -> int:
    return int(lib().flint_moe_launch_count(h))


def flint_moe_forward_launches(h: int, T: int) -> int:
    return int(lib().flint_moe_forward_launches(h, T))


def flint_moe_debug_act_quant(x, T: int, K: int, codes, scales, rowscale, stream=None) -> None:
    _check(lib().flint_moe_debug_act_quant(_ptr(x), T, K, _ptr(codes), _ptr(scales), _ptr(rowscale), _stream(stream)),
           "flint_moe_debug_act_quant")


def flint_moe_debug_fp4_gemm(a_codes, a_scales, b_codes, b_scales, M: int, N: int, K: int, d, stream=None) -> None:
    _check(lib().flint_moe_debug_fp4_gemm(_ptr(a_codes), _ptr(a_scales), _ptr(b_codes), _ptr(b_scales), M, N, K,
                                          _ptr(d), _stream(stream)), "flint_moe_debug_fp4_gemm")


def flint_moe_tensor_core_plan(h: int, layer: int, T: int) -> int:
    return int(lib().flint_moe_tensor_core_plan(h, layer, T))


def flint_moe_profile_begin(h: int, max_forwards: int) -> None:
    _check(lib().flint_moe_profile_begin(h, max_forwards), "flint_moe_profile_begin")


PROFILE_PHASES = ("router_topk_bucket", "gateup", "down_combine", "act_quant", "combine_out")


def flint_moe_profile_end(h: int):
    """-> (per-phase summed milliseconds in PROFILE_PHASES order, forwards)."""
    ms = (ctypes.c_float * len(PROFILE_PHASES))()
    n = _I()
    _check(lib().flint_moe_profile_end(h, ms, ctypes.byref(n)), "flint_moe_profile_end")
    return [float(v) for v in ms], int(n.value)


def flint_moe_load_lm_head(h: int, codes: np.ndarray, scales: np.ndarray, tensor_scale: float) -> None:
    """Host arrays in the canonical layout: codes uint8 [vocab, d/2], scales uint8 [vocab, d/16]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    _check(lib().flint_moe_load_lm_head(h, codes.shape[0], codes.ctypes.data, scales.ctypes.data,
                                        float(tensor_scale)), "flint_moe_load_lm_head")


def flint_moe_lm_head(h: int, hidden, T: int, logits, stream=None) -> None:
    _check(lib().flint_moe_lm_head(h, _ptr(hidden), T, _ptr(logits), _stream(stream)), "flint_moe_lm_head")


def flint_moe_sample(h: int, logits, T: int, temperature: float, top_k: int, top_p: float, u, tokens, topk=None,
                     stream=None) -> None:
    _check(lib().flint_moe_sample(h, _ptr(logits), T, float(temperature), top_k, float(top_p), _ptr(u),
                                  _ptr(tokens), _ptr(topk), _stream(stream)), "flint_moe_sample")


def flint_moe_probe_fp4_peak(n: int, iters: int) -> tuple[float, float]:
    """(milliseconds, FLOPs) of the dense FP4 tensor-core probe on the current device."""
    ms = ctypes.c_float(0.0)
    flops = ctypes.c_double(0.0)
    _check(lib().flint_moe_probe_fp4_peak(n, iters, ctypes.byref(ms), ctypes.byref(flops)), "flint_moe_probe_fp4_peak")
    return float(ms.value), float(flops.value)


def flint_moe_attn_decode(n_heads: int, n_kv: int, window: int, cap: int, rope: bool, B: int, q, k, v, k_cache, v_cache,
                      pos, q_norm_w, k_norm_w, sinks, out, rope_theta: float = 10000.0, eps: float = 1e-6,
                      stream=None) -> None:
    cfg = flint_moe_attn_config(n_heads, n_kv, 128, window, cap, 1 if rope else 0, rope_theta, eps)
    _check(lib().flint_moe_attn_decode(ctypes.byref(cfg), B, _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(pos), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(sinks), _ptr(out),
                                   _stream(stream)), "flint_moe_attn_decode")


def flint_moe_quantize_nvfp4(w, R: int, K: int, codes, scales, tensor_scale, stream=None) -> None:
    _check(lib().flint_moe_quantize_nvfp4(_ptr(w), R, K, _ptr(codes), _ptr(scales), _ptr(tensor_scale),
                                          _stream(stream)), "flint_moe_quantize_nvfp4")


def flint_moe_debug_wait_timeout(h: int, kind: int, spin_limit: int, stream=None) -> None:
    _check(lib().flint_moe_debug_wait_timeout(h, kind, spin_limit, _stream(stream)), "flint_moe_debug_wait_timeout")


def flint_moe_bucket_noalloc(idx, T: int, k: int, E: int, offsets, perm, stream=None) -> None:
    """Bucketing without a handle and without allocating (static scratch in the
    library; see include/flint_moe.h for its limits and sharing rules)."""
    fn = lib().flint_moe_bucket_noalloc
    fn.restype = _I
    fn.argtypes = [_P, _I, _I, _I, _P, _P, _P]
    _check(fn(_ptr(idx), T, k, E, _ptr(offsets), _ptr(perm), _stream(stream)), "flint_moe_bucket_noalloc")


# ---------------------------------------------------------------------------
# convenience object
# ---------------------------------------------------------------------------


class MoE:
    """A handle plus torch-side buffers. `layers` are canonical host weights
    (objects with router, router_bias, codes, scales, tensor_scale)."""

    def __init__(self, cfg, max_tokens: int, n_layers: int = 1, device: int = 0):
        import torch
        self.cfg = cfg
        self.device = torch.device("cuda", device)
        self.h = flint_moe_create(cfg.d, cfg.f, cfg.n_experts, cfg.top_k, 1, cfg.wfmt, max_tokens,
                                  n_layers, device)

    def load(self, layer: int, w) -> None:
        flint_moe_load_weights(self.h, layer, w.router, w.router_bias, w.codes, w.scales,
                               w.tensor_scale if self.cfg.wfmt == FLINT_W_NVFP4 else None)

    def forward(self, hidden, layer: int = 0, out=None, stream=None):
        import torch
        T = hidden.shape[0]
        if out is None:
            out = torch.empty_like(hidden)
        flint_moe_forward(self.h, layer, hidden, T, out, stream)
        return out

    def forward_stack(self, hidden, layer0: int, n_layers: int, stream=None):
        flint_moe_forward_stack(self.h, layer0, n_layers, hidden, hidden.shape[0], stream)
        return hidden

    def close(self) -> None:
        if self.h:
            flint_moe_destroy(self.h)
            self.h = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def hidden_to_device(bits: np.ndarray, device: int = 0):
    """bf16 bit patterns (uint16 [T, d]) -> torch bfloat16 CUDA tensor."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(f"cuda:{device}")
    return t.view(torch.bfloat16)


def hidden_to_host(t) -> np.ndarray:
    """torch bfloat16 tensor -> bf16 bit patterns uint16."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
