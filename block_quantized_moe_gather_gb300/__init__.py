"""Python binding of the block-quantized MoE gather-qmm library (``libbq.so``).

Argument marshalling only: every function forwards device pointers of
PyTorch tensors and the current CUDA stream to the C ABI declared in
``include/bq.h``.  All arithmetic runs in the library's CUDA kernels; there
is no CPU fallback.  Importing this package fails when the library has not
been built (``python block_quantized_moe_gather_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_size_t, c_uint64, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python block_quantized_moe_gather_gb300/build.py`")
_lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------- constants
OK = 0
FMT_Q8_0, FMT_Q2_K, FMT_INT4_G64, FMT_MXFP4, FMT_FP8_B128 = 1, 2, 3, 4, 5
FMT_BY_NAME = {"q8_0": FMT_Q8_0, "q2_k": FMT_Q2_K, "int4": FMT_INT4_G64, "mxfp4": FMT_MXFP4,
               "fp8_b128": FMT_FP8_B128}
DEV_OK, DEV_BAD_EXPERT_ID, DEV_WAIT_TIMEOUT, DEV_SCALE_RANGE = 0, 1, 2, 3
STATUS_NAMES = {0: "BQ_OK", 1: "BQ_ERR_NULL", 2: "BQ_ERR_SHAPE", 3: "BQ_ERR_ALIGN", 4: "BQ_ERR_FORMAT",
                5: "BQ_ERR_WORKSPACE", 6: "BQ_ERR_CUDA", 7: "BQ_ERR_DEVICE", 8: "BQ_ERR_ARCH"}


class QWeightC(ctypes.Structure):
    _fields_ = [("fmt", c_int32), ("n_mats", c_int32), ("n", c_int32), ("k", c_int32),
                ("swiglu", c_int32), ("reserved", c_int32), ("data", c_void_p)]


class MoEDescC(ctypes.Structure):
    _fields_ = [("T", c_int32), ("hidden", c_int32), ("inter", c_int32), ("n_experts", c_int32),
                ("topk", c_int32), ("scoring", c_int32), ("w_gate_up", QWeightC), ("w_down", QWeightC),
                ("shared_gate_up", POINTER(QWeightC)), ("shared_down", POINTER(QWeightC)),
                ("route_scale", c_float), ("reserved", c_int32)]


_SIGS = {
    "bq_status_string": (c_char_p, [c_int32]),
    "bq_last_error": (c_char_p, []),
    "bq_device_status": (c_int32, [c_void_p, POINTER(c_int32)]),
    "bq_gguf_dequant_q8_0": (c_int32, [c_void_p, c_int64, c_void_p, c_void_p]),
    "bq_gguf_dequant_q2_k": (c_int32, [c_void_p, c_int64, c_void_p, c_void_p]),
    "bq_dequant_mxfp4": (c_int32, [c_void_p, c_int64, c_void_p, c_void_p]),
    "bq_dequant_fp8_b128": (c_int32, [c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "bq_qweight_bytes": (c_size_t, [c_int32, c_int32, c_int32, c_int32]),
    "bq_repack_q8_0": (c_int32, [c_void_p, POINTER(QWeightC), c_void_p]),
    "bq_repack_q2_k": (c_int32, [c_void_p, POINTER(QWeightC), c_void_p]),
    "bq_repack_int4": (c_int32, [c_void_p, c_void_p, c_void_p, POINTER(QWeightC), c_void_p]),
    "bq_repack_mxfp4": (c_int32, [c_void_p, POINTER(QWeightC), c_void_p]),
    "bq_repack_fp8_b128": (c_int32, [c_void_p, c_void_p, POINTER(QWeightC), c_void_p]),
    "bq_qmm": (c_int32, [c_void_p, c_int32, POINTER(QWeightC), c_void_p, c_void_p]),
    "bq_moe_route": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p]),
    "bq_moe_route_scored": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_float, c_void_p,
                                      c_void_p, c_void_p]),
    "bq_moe_permute_workspace_bytes": (c_size_t, [c_int32, c_int32, c_int32]),
    "bq_moe_permute": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_size_t, c_void_p]),
    "bq_moe_workspace_bytes": (c_size_t, [POINTER(MoEDescC)]),
    "bq_moe_permute_noalloc": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p]),
    "bq_set_stage_events": (c_int32, [c_int32, c_void_p, c_void_p]),
    "bq_rmsnorm": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_float, c_void_p, c_void_p]),
    "bq_rmsnorm_qmm": (c_int32, [c_void_p, c_int32, c_void_p, c_float, POINTER(QWeightC), c_void_p, c_void_p,
                                 c_void_p]),
    "bq_moe_hidden_workspace_bytes": (c_size_t, [POINTER(MoEDescC)]),
    "bq_moe_gather_qmm_hidden": (c_int32, [POINTER(MoEDescC), POINTER(QWeightC), c_void_p, c_void_p, c_float,
                                           c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "bq_launch_count": (c_uint64, []),
    "bq_test_set_wait_probe": (c_int32, [c_int32, c_uint64]),
    "bq_moe_gather_qmm": (c_int32, [POINTER(MoEDescC), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_size_t, c_void_p]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class BQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.bq_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")


def _check(status: int, where: str):
    if status != OK:
        raise BQError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def status_string(s: int) -> str:
    return _lib.bq_status_string(s).decode()


def last_error() -> str:
    return _lib.bq_last_error().decode()


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status code."""
    code = c_int32(0)
    st = _lib.bq_device_status(_stream(stream), ctypes.byref(code))
    if st not in (OK, 7):
        raise BQError(st, "bq_device_status")
    return code.value


# ---------------------------------------------------------------- dequant
def gguf_dequant_q8_0(blocks, out, stream=None):
    """blocks: uint8 device tensor of n*34 bytes; out: fp32 device tensor of n*32."""
    n = blocks.numel() // 34
    _check(_lib.bq_gguf_dequant_q8_0(_ptr(blocks), n, _ptr(out), _stream(stream)), "bq_gguf_dequant_q8_0")
    return out


def gguf_dequant_q2_k(blocks, out, stream=None):
    n = blocks.numel() // 84
    _check(_lib.bq_gguf_dequant_q2_k(_ptr(blocks), n, _ptr(out), _stream(stream)), "bq_gguf_dequant_q2_k")
    return out


def dequant_mxfp4(blocks, out, stream=None):
    """blocks: uint8 device tensor of n*17 bytes; out: fp32 device tensor of n*32."""
    n = blocks.numel() // 17
    _check(_lib.bq_dequant_mxfp4(_ptr(blocks), n, _ptr(out), _stream(stream)), "bq_dequant_mxfp4")
    return out


def dequant_fp8_b128(weight, scales, out, stream=None):
    """weight: uint8 device tensor [n, k] (e4m3 bytes); scales: fp32 [ceil(n/128), ceil(k/128)];
    out: fp32 [n, k]."""
    n, k = weight.shape
    _check(_lib.bq_dequant_fp8_b128(_ptr(weight), _ptr(scales), n, k, _ptr(out), _stream(stream)),
           "bq_dequant_fp8_b128")
    return out


# ---------------------------------------------------------------- weights
def qweight_bytes(fmt: int, n_mats: int, n: int, k: int) -> int:
    return int(_lib.bq_qweight_bytes(fmt, n_mats, n, k))


class QWeight:
    """A repacked quantised weight stack [n_mats][n][k] held in a device
    uint8 tensor (``buf``), plus the C descriptor pointing at it."""

    def __init__(self, fmt: int, n_mats: int, n: int, k: int, swiglu: bool = False, device="cuda"):
        import torch
        nbytes = qweight_bytes(fmt, n_mats, n, k)
        if nbytes == 0:
            raise BQError(2, f"QWeight(fmt={fmt}, {n_mats}x{n}x{k})")
        # 256-byte alignment: the caching allocator returns 512-byte aligned blocks
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.fmt, self.n_mats, self.n, self.k, self.swiglu = fmt, n_mats, n, k, int(swiglu)
        self.c = QWeightC(fmt, n_mats, n, k, int(swiglu), 0, self.buf.data_ptr())

    @property
    def nbytes(self) -> int:
        return self.buf.numel()


def repack_q8_0(blocks, w: QWeight, stream=None) -> QWeight:
    _check(_lib.bq_repack_q8_0(_ptr(blocks), ctypes.byref(w.c), _stream(stream)), "bq_repack_q8_0")
    return w


def repack_q2_k(blocks, w: QWeight, stream=None) -> QWeight:
    _check(_lib.bq_repack_q2_k(_ptr(blocks), ctypes.byref(w.c), _stream(stream)), "bq_repack_q2_k")
    return w


def repack_int4(words, scales, biases, w: QWeight, stream=None) -> QWeight:
    _check(_lib.bq_repack_int4(_ptr(words), _ptr(scales), _ptr(biases), ctypes.byref(w.c), _stream(stream)),
           "bq_repack_int4")
    return w


def repack_mxfp4(blocks, w: QWeight, stream=None) -> QWeight:
    _check(_lib.bq_repack_mxfp4(_ptr(blocks), ctypes.byref(w.c), _stream(stream)), "bq_repack_mxfp4")
    return w


def repack_fp8_b128(weight, scales, w: QWeight, stream=None) -> QWeight:
    _check(_lib.bq_repack_fp8_b128(_ptr(weight), _ptr(scales), ctypes.byref(w.c), _stream(stream)),
           "bq_repack_fp8_b128")
    return w


# ---------------------------------------------------------------- compute
def qmm(x, w: QWeight, y, stream=None):
    """y[m][n] = x[m][k] W^T; x fp16 [m, k], y fp32 [m, n] (device)."""
    m = x.shape[0] if x.dim() == 2 else 1
    _check(_lib.bq_qmm(_ptr(x), m, ctypes.byref(w.c), _ptr(y), _stream(stream)), "bq_qmm")
    return y


def moe_route(logits, bias, k: int, ids, weights, stream=None):
    t, e = logits.shape
    _check(_lib.bq_moe_route(_ptr(logits), _ptr(bias), t, e, k, _ptr(ids), _ptr(weights), _stream(stream)),
           "bq_moe_route")


# bq_scoring
SCORE_SOFTMAX, SCORE_SOFTMAX_THEN_BIAS, SCORE_SQRTSOFTPLUS = 0, 1, 2
SCORING_BY_NAME = {"softmax": SCORE_SOFTMAX, "softmax_then_bias": SCORE_SOFTMAX_THEN_BIAS,
                   "sqrtsoftplus": SCORE_SQRTSOFTPLUS}


def moe_route_scored(logits, bias, k: int, scoring: int, scale: float, ids, weights, stream=None):
    t, e = logits.shape
    _check(_lib.bq_moe_route_scored(_ptr(logits), _ptr(bias), t, e, k, scoring, scale, _ptr(ids), _ptr(weights),
                                    _stream(stream)),
           "bq_moe_route_scored")


def moe_permute_workspace_bytes(t: int, k: int, e: int) -> int:
    return int(_lib.bq_moe_permute_workspace_bytes(t, k, e))


def moe_permute(ids, n_experts: int, counts, offsets, perm_token, perm_slot, inv, workspace, stream=None):
    t, k = ids.shape
    _check(_lib.bq_moe_permute(_ptr(ids), t, k, n_experts, _ptr(counts), _ptr(offsets), _ptr(perm_token),
                               _ptr(perm_slot), _ptr(inv), _ptr(workspace), workspace.numel(), _stream(stream)),
           "bq_moe_permute")


STAGE_ROUTE_PERMUTE, STAGE_GATE_UP, STAGE_DOWN, STAGE_SHARED, STAGE_COMBINE, STAGE_NORM_ROUTER = range(6)


def set_stage_events(stage: int, start=None, stop=None):
    """Have later layer calls record `start`/`stop` (torch.cuda.Event, already
    recorded once so that they exist) around one stage; None clears."""
    h = (lambda ev: None if ev is None else ctypes.c_void_p(ev.cuda_event))
    _check(_lib.bq_set_stage_events(stage, h(start), h(stop)), "bq_set_stage_events")


def launch_count() -> int:
    return int(_lib.bq_launch_count())


def test_set_wait_probe(skip_weight_copies: bool, wait_limit_ns: int = 0):
    """Test hook: GEMM launches that follow take `wait_limit_ns` as the bound of
    their barrier waits and, with `skip_weight_copies`, issue no weight copies
    (so those waits run out); (False, 0) restores the defaults."""
    _check(_lib.bq_test_set_wait_probe(int(bool(skip_weight_copies)), int(wait_limit_ns)),
           "bq_test_set_wait_probe")


def moe_permute_noalloc(ids, n_experts: int, counts, offsets, perm_token, perm_slot, inv, stream=None):
    """bq_moe_permute without a workspace: for callers that cannot allocate
    device memory at call time.  Scratch is a fixed array built into the
    library (limit: ceil(T*k/256) * E <= 65536); calls that overlap on the
    GPU race on it."""
    t, k = ids.shape
    _check(_lib.bq_moe_permute_noalloc(_ptr(ids), t, k, n_experts, _ptr(counts), _ptr(offsets), _ptr(perm_token),
                                       _ptr(perm_slot), _ptr(inv), _stream(stream)),
           "bq_moe_permute_noalloc")


class MoELayer:
    """Descriptor of one MoE layer over repacked weights (host struct)."""

    def __init__(self, t: int, hidden: int, inter: int, n_experts: int, topk: int, w_gate_up: QWeight,
                 w_down: QWeight, shared_gate_up: QWeight | None = None, shared_down: QWeight | None = None,
                 scoring: int = 0, route_scale: float = 1.0):
        self.weights = (w_gate_up, w_down, shared_gate_up, shared_down)  # keep buffers alive
        self._s_gu = shared_gate_up.c if shared_gate_up else None
        self._s_d = shared_down.c if shared_down else None
        self.c = MoEDescC(t, hidden, inter, n_experts, topk, scoring, w_gate_up.c, w_down.c,
                          ctypes.pointer(self._s_gu) if self._s_gu else None,
                          ctypes.pointer(self._s_d) if self._s_d else None, route_scale, 0)

    def set_tokens(self, t: int):
        self.c.T = t

    def workspace_bytes(self) -> int:
        return int(_lib.bq_moe_workspace_bytes(ctypes.byref(self.c)))

    def hidden_workspace_bytes(self) -> int:
        """Workspace of moe_gather_qmm_hidden (layer + normalised x + logits)."""
        return int(_lib.bq_moe_hidden_workspace_bytes(ctypes.byref(self.c)))


def moe_workspace_bytes(layer: MoELayer) -> int:
    return layer.workspace_bytes()


def moe_gather_qmm(layer: MoELayer, x, router_logits, logit_bias, y, workspace, stream=None):
    _check(_lib.bq_moe_gather_qmm(ctypes.byref(layer.c), _ptr(x), _ptr(router_logits), _ptr(logit_bias),
                                  _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)),
           "bq_moe_gather_qmm")
    return y


# ---------------------------------------------------------------- RMSNorm, fused
def rmsnorm(h, gamma, eps: float, x, stream=None):
    """x = gamma * h / sqrt(mean(h^2) + eps) per row; h, x fp16 [T, H], gamma fp16 [H]."""
    t, hdim = h.shape
    _check(_lib.bq_rmsnorm(_ptr(h), t, hdim, _ptr(gamma), eps, _ptr(x), _stream(stream)), "bq_rmsnorm")
    return x


def rmsnorm_qmm(h, gamma, eps: float, w: QWeight, y, x_out=None, stream=None):
    """y = W rmsnorm(h) (fp32 [m, n]); x_out (fp16 [m, k]) receives the normalised
    rows (required for m > 8)."""
    m = h.shape[0]
    _check(_lib.bq_rmsnorm_qmm(_ptr(h), m, _ptr(gamma), eps, ctypes.byref(w.c), _ptr(x_out), _ptr(y),
                               _stream(stream)),
           "bq_rmsnorm_qmm")
    return y


def moe_gather_qmm_hidden(layer: MoELayer, router: QWeight, hidden, gamma, eps: float, logit_bias, y, workspace,
                          stream=None):
    """The MoE layer from hidden states: RMSNorm + router matmul, then moe_gather_qmm."""
    _check(_lib.bq_moe_gather_qmm_hidden(ctypes.byref(layer.c), ctypes.byref(router.c), _ptr(hidden), _ptr(gamma),
                                         eps, _ptr(logit_bias), _ptr(y), _ptr(workspace), workspace.numel(),
                                         _stream(stream)),
           "bq_moe_gather_qmm_hidden")
    return y
