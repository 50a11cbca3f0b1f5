"""ctypes binding of libmoeblock.so (include/moe_block.h). Argument marshalling only: every step of the block
runs in the library's CUDA kernels; torch supplies device memory and streams. A missing library raises."""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoeblock.so")

MOE_OK = 0
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_NOT_LOADED",
          -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE_TIMEOUT", -6: "MOE_ERR_NO_DEVICE"}

WEIGHT_FIELDS = [
    "router_q", "router_s", "router_b", "exp_gate_q", "exp_gate_s", "exp_gate_b", "exp_up_q", "exp_up_s",
    "exp_up_b", "exp_down_q", "exp_down_s", "exp_down_b", "sh_gate_q", "sh_gate_s", "sh_gate_b", "sh_up_q",
    "sh_up_s", "sh_up_b", "sh_down_q", "sh_down_s", "sh_down_b", "rms_gamma",
]
EXPORTS = ["moe_block_create", "moe_block_load_weights", "moe_block_forward", "moe_block_forward_host",
           "moe_block_forward_residual", "moe_block_get_status", "moe_block_destroy", "moe_block_strerror",
           "moe_last_cuda_error", "moe_block_debug_dequant", "moe_block_debug_last_routing",
           "moe_block_debug_set_wait", "moe_block_debug_set_trace", "moe_block_last_launch_count",
           "moe_router_topk_noalloc", "moe_debug_decode_plan", "moe_stack_create", "moe_stack_load_layer",
           "moe_stack_forward", "moe_stack_get_status", "moe_stack_layer", "moe_stack_destroy",
           "moe_affine_convert", "moe_affine_free", "moe_block_load_affine"]


class MoeError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        lib = _LIB
        extra = ""
        if lib is not None and status == -4:
            extra = " (" + lib.moe_last_cuda_error().decode() + ")"
        super().__init__(f"{what}: {STATUS.get(status, status)}{extra}")


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("expert_inter", ctypes.c_int), ("shared_inter", ctypes.c_int), ("group_size", ctypes.c_int),
                ("max_tokens", ctypes.c_int)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class AffineTensor(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("bits", ctypes.c_int)]


AFFINE_TENSORS = ["router", "exp_gate", "exp_up", "exp_down", "sh_gate", "sh_up", "sh_down"]


class AffineWeights(ctypes.Structure):
    _fields_ = [(n, AffineTensor) for n in AFFINE_TENSORS] + [
        ("shared_gate", ctypes.c_void_p), ("rms_gamma", ctypes.c_void_p), ("scale_dtype", ctypes.c_int)]


DTYPES = {"f16": 0, "bf16": 1}


def _affine_struct(aff: dict):
    """An AffineWeights struct over host numpy arrays: aff[name] = (q uint32, scales uint16, biases uint16, bits)
    for every name of AFFINE_TENSORS, aff["shared_gate"] uint16, aff["rms_gamma"] uint16 or absent,
    aff["scale_dtype"] "f16" or "bf16". Returns the struct and the arrays it points into."""
    keep = []
    A = AffineWeights()

    def ptr(a, dtype):
        a = np.ascontiguousarray(a).view(dtype)
        keep.append(a)
        return a.ctypes.data

    for n in AFFINE_TENSORS:
        q, s, b, bits = aff[n]
        setattr(A, n, AffineTensor(ptr(q, np.uint32), ptr(s, np.uint16), ptr(b, np.uint16), int(bits)))
    A.shared_gate = ptr(aff["shared_gate"], np.uint16)
    A.rms_gamma = ptr(aff["rms_gamma"], np.uint16) if aff.get("rms_gamma") is not None else None
    A.scale_dtype = DTYPES[aff["scale_dtype"]]
    return A, keep


def affine_convert(cfg, aff: dict):
    """The library's conversion of affine-layout host arrays (see _affine_struct) into the canonical layout: a
    dict of numpy arrays (codes uint8, fp16 pairs as float16), copied out of the library's buffers. Host only."""
    lib = load_library()
    A, keep = _affine_struct(aff)
    c = Config(cfg.hidden, cfg.n_experts, cfg.top_k, cfg.expert_inter, cfg.shared_inter, 64, 1)
    W = Weights()
    _check(lib.moe_affine_convert(ctypes.byref(c), ctypes.byref(A), ctypes.byref(W)), "moe_affine_convert")
    H, E, I, Is = cfg.hidden, cfg.n_experts, cfg.expert_inter, cfg.shared_inter
    shapes = {"router": ((E + 1, H), (E + 1, H // 64)), "exp_gate": ((E, I, H // 2), (E, I, H // 64)),
              "exp_up": ((E, I, H // 2), (E, I, H // 64)), "exp_down": ((E, H, I // 2), (E, H, I // 64)),
              "sh_gate": ((Is, H), (Is, H // 64)), "sh_up": ((Is, H), (Is, H // 64)), "sh_down": ((H, Is), (H, Is // 64))}
    out = {}
    try:
        for n, (qs, ss) in shapes.items():
            out[n + "_q"] = np.ctypeslib.as_array(ctypes.cast(getattr(W, n + "_q"), ctypes.POINTER(ctypes.c_uint8)),
                                                  shape=qs).copy()
            for sfx in ("_s", "_b"):
                a = np.ctypeslib.as_array(ctypes.cast(getattr(W, n + sfx), ctypes.POINTER(ctypes.c_uint16)), shape=ss)
                out[n + sfx] = a.copy().view(np.float16)
    finally:
        lib.moe_affine_free(ctypes.byref(W))
    return out


_LIB = None


def load_library(path: str = LIB_PATH):
    """Load libmoeblock.so (built by w4a16_top_mixture_gb300.build). Raises if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m w4a16_top_mixture_gb300.build` "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    vp, i, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32
    lib.moe_block_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(vp)]
    lib.moe_block_load_weights.argtypes = [vp, ctypes.POINTER(Weights), i, vp]
    lib.moe_block_forward.argtypes = [vp, vp, vp, i, vp]
    lib.moe_block_forward_host.argtypes = [vp, vp, vp, i, vp]
    lib.moe_block_forward_residual.argtypes = [vp, vp, vp, i, ctypes.c_float, vp]
    lib.moe_block_get_status.argtypes = [vp, ctypes.POINTER(u32)]
    lib.moe_block_destroy.argtypes = [vp]
    lib.moe_block_destroy.restype = None
    lib.moe_block_strerror.argtypes = [i]
    lib.moe_block_strerror.restype = ctypes.c_char_p
    lib.moe_last_cuda_error.argtypes = []
    lib.moe_last_cuda_error.restype = ctypes.c_char_p
    lib.moe_block_debug_dequant.argtypes = [vp, i, i, vp, vp]
    lib.moe_block_debug_last_routing.argtypes = [vp, i, vp, vp, vp, vp, vp]
    lib.moe_block_debug_set_wait.argtypes = [vp, u32, i]
    lib.moe_block_last_launch_count.argtypes = [vp]
    lib.moe_block_debug_set_trace.argtypes = [vp, vp]
    lib.moe_router_topk_noalloc.argtypes = [vp, vp, vp, i, i, i, vp, i, vp, vp, vp, vp]
    lib.moe_debug_decode_plan.argtypes = [ctypes.POINTER(Config), i, i, i, ctypes.POINTER(ctypes.c_int32)]
    lib.moe_stack_create.argtypes = [ctypes.POINTER(Config), i, ctypes.c_float, ctypes.POINTER(vp)]
    lib.moe_affine_convert.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(AffineWeights), ctypes.POINTER(Weights)]
    lib.moe_affine_free.argtypes = [ctypes.POINTER(Weights)]
    lib.moe_affine_free.restype = None
    lib.moe_block_load_affine.argtypes = [vp, ctypes.POINTER(AffineWeights), vp]
    lib.moe_stack_load_layer.argtypes = [vp, i, ctypes.POINTER(Weights), i, vp]
    lib.moe_stack_forward.argtypes = [vp, vp, vp, i, vp, vp]
    lib.moe_stack_get_status.argtypes = [vp, ctypes.POINTER(u32)]
    lib.moe_stack_layer.argtypes = [vp, i]
    lib.moe_stack_layer.restype = vp
    lib.moe_stack_destroy.argtypes = [vp]
    lib.moe_stack_destroy.restype = None
    for n in EXPORTS:
        if not hasattr(lib, n):
            raise RuntimeError(f"{path} does not export {n}")
    _LIB = lib
    return lib


def decode_plan(cfg, T, num_sms, max_smem):
    """Host-only query of the fused decode kernel's launch plan (no device needed): (status, plan), plan a dict
    of grid, smem, stages, stage_bytes, h_staged when status == 0."""
    lib = load_library()
    c = Config(cfg.hidden, cfg.n_experts, cfg.top_k, cfg.expert_inter, cfg.shared_inter, 64, 16)
    out = (ctypes.c_int32 * 5)()
    st = lib.moe_debug_decode_plan(ctypes.byref(c), int(T), int(num_sms), int(max_smem), out)
    if st != MOE_OK:
        return st, None
    return st, dict(zip(("grid", "smem", "stages", "stage_bytes", "h_staged"), list(out)))


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


class MoeBlock:
    """One block's weights on the current CUDA device, and its forward entry points."""

    def __init__(self, hidden=2048, n_experts=256, top_k=8, expert_inter=512, shared_inter=512, max_tokens=16):
        self.lib = load_library()
        self.cfg = Config(hidden, n_experts, top_k, expert_inter, shared_inter, 64, max_tokens)
        h = ctypes.c_void_p()
        _check(self.lib.moe_block_create(ctypes.byref(self.cfg), ctypes.byref(h)), "moe_block_create")
        self.h = h
        self.hidden, self.n_experts, self.top_k = hidden, n_experts, top_k
        self.max_tokens = max_tokens

    @classmethod
    def from_config(cls, cfg, max_tokens=16):
        return cls(cfg.hidden, cfg.n_experts, cfg.top_k, cfg.expert_inter, cfg.shared_inter, max_tokens)

    @classmethod
    def borrow(cls, stack, layer):
        """The block handle of one layer of a MoeStack (owned by the stack: close() leaves it alone)."""
        b = cls.__new__(cls)
        b.lib = stack.lib
        b.cfg = stack.cfg
        b.h = None
        b._borrowed = ctypes.c_void_p(stack.lib.moe_stack_layer(stack.h, int(layer)))
        b.hidden, b.n_experts, b.top_k = stack.cfg.hidden, stack.cfg.n_experts, stack.cfg.top_k
        b.max_tokens = stack.cfg.max_tokens
        b._stack = stack
        return b

    @property
    def handle(self):
        return self.h if self.h is not None else getattr(self, "_borrowed", None)

    def close(self):
        if getattr(self, "h", None):
            self.lib.moe_block_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_weights(self, w: dict, stream=None):
        """w: canonical arrays (numpy on the host, or torch tensors on the device; fp16 as float16/uint16)."""
        W, keep, on_dev = _weights_struct(w)
        _check(self.lib.moe_block_load_weights(self.handle, ctypes.byref(W), int(on_dev), _stream_ptr(stream)),
               "moe_block_load_weights")

    def load_affine(self, aff: dict, stream=None):
        """aff: host arrays in the affine checkpoint layout (see _affine_struct)."""
        A, keep = _affine_struct(aff)
        _check(self.lib.moe_block_load_affine(self.handle, ctypes.byref(A), _stream_ptr(stream)),
               "moe_block_load_affine")

    def forward(self, x, out=None, stream=None):
        import torch
        assert x.dtype == torch.float16 and x.is_cuda and x.is_contiguous()
        if out is None:
            out = torch.empty_like(x)
        T = x.shape[0] if x.dim() == 2 else 0
        _check(self.lib.moe_block_forward(self.handle, _ptr(x), _ptr(out), T, _stream_ptr(stream)), "moe_block_forward")
        return out

    def forward_residual(self, h_in, h_out=None, eps=1e-6, stream=None):
        import torch
        assert h_in.dtype == torch.float16 and h_in.is_cuda and h_in.is_contiguous()
        if h_out is None:
            h_out = torch.empty_like(h_in)
        _check(self.lib.moe_block_forward_residual(self.handle, _ptr(h_in), _ptr(h_out), h_in.shape[0], float(eps),
                                                   _stream_ptr(stream)), "moe_block_forward_residual")
        return h_out

    def forward_host(self, x_host, out_host=None, stream=None):
        """x_host: numpy/pinned-torch fp16 [T, H] on the host; returns the host output."""
        import torch
        if isinstance(x_host, np.ndarray):
            x_host = torch.from_numpy(np.ascontiguousarray(x_host))
        if out_host is None:
            out_host = torch.empty_like(x_host)
        _check(self.lib.moe_block_forward_host(self.handle, _ptr(x_host), _ptr(out_host), x_host.shape[0],
                                               _stream_ptr(stream)), "moe_block_forward_host")
        return out_host

    def status(self):
        f = ctypes.c_uint32(0)
        s = self.lib.moe_block_get_status(self.handle, ctypes.byref(f))
        return s, f.value

    def debug_dequant(self, which, index=0, stream=None):
        import torch
        H, E, I, Is = self.cfg.hidden, self.cfg.n_experts, self.cfg.expert_inter, self.cfg.shared_inter
        shape = {0: (E + 1, H), 1: (I, H), 2: (I, H), 3: (H, I), 4: (Is, H), 5: (Is, H), 6: (H, Is)}[which]
        out = torch.empty(shape, dtype=torch.float32, device="cuda")
        _check(self.lib.moe_block_debug_dequant(self.handle, which, index, _ptr(out), _stream_ptr(stream)),
               "moe_block_debug_dequant")
        return out

    def last_routing(self, T, stream=None):
        import torch
        E, K = self.cfg.n_experts, self.cfg.top_k
        lg = torch.empty((T, E + 1), dtype=torch.float32, device="cuda") if T <= 16 else None
        ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        sg = torch.empty((T,), dtype=torch.float32, device="cuda")
        _check(self.lib.moe_block_debug_last_routing(self.handle, T, _ptr(lg), _ptr(ids), _ptr(w), _ptr(sg),
                                                     _stream_ptr(stream)), "moe_block_debug_last_routing")
        return {"logits": lg, "ids": ids, "w": w, "sg": sg}

    def set_wait(self, timeout_us=0, skip_arrive=False):
        _check(self.lib.moe_block_debug_set_wait(self.handle, int(timeout_us), int(bool(skip_arrive))), "set_wait")

    def set_trace(self, buf=None):
        """buf: int64 CUDA tensor of >= 96 * SM-count entries, or None to stop tracing."""
        if buf is not None:
            import torch
            sms = torch.cuda.get_device_properties(buf.device).multi_processor_count
            if buf.dtype != torch.int64 or buf.numel() < 96 * sms or not buf.is_contiguous():
                raise ValueError(f"trace buffer must be a contiguous int64 tensor of >= {96 * sms} entries")
        _check(self.lib.moe_block_debug_set_trace(self.handle, _ptr(buf)), "set_trace")

    def last_launch_count(self):
        return self.lib.moe_block_last_launch_count(self.handle)


def _weights_struct(w: dict):
    """A Weights struct over the canonical arrays of w (all numpy on the host, or all torch tensors on the device),
    with the objects that must stay alive while the library reads them, and whether they are on the device."""
    import torch
    keep = []
    on_dev = None
    W = Weights()
    for n in WEIGHT_FIELDS:
        a = w.get(n)
        if a is None:
            continue
        if isinstance(a, np.ndarray):
            a = np.ascontiguousarray(a)
            if on_dev:
                raise ValueError("mix of host and device weights")
            on_dev = False
            keep.append(a)
            setattr(W, n, a.ctypes.data)
        else:
            assert isinstance(a, torch.Tensor) and a.is_cuda and a.is_contiguous()
            if on_dev is False:
                raise ValueError("mix of host and device weights")
            on_dev = True
            keep.append(a)
            setattr(W, n, a.data_ptr())
    return W, keep, bool(on_dev)


class MoeStack:
    """n_layers blocks of one shape, h_{l+1} = h_l + block_l(RMSNorm_l(h_l)), run as one chain of launches."""

    def __init__(self, cfg, n_layers, max_tokens=1, eps=1e-6):
        self.lib = load_library()
        self.cfg = Config(cfg.hidden, cfg.n_experts, cfg.top_k, cfg.expert_inter, cfg.shared_inter, 64, max_tokens)
        h = ctypes.c_void_p()
        _check(self.lib.moe_stack_create(ctypes.byref(self.cfg), int(n_layers), float(eps), ctypes.byref(h)),
               "moe_stack_create")
        self.h = h
        self.n_layers = n_layers
        self.hidden = cfg.hidden

    def close(self):
        if getattr(self, "h", None):
            self.lib.moe_stack_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_layer(self, layer, w: dict, stream=None):
        W, keep, on_dev = _weights_struct(w)
        _check(self.lib.moe_stack_load_layer(self.h, int(layer), ctypes.byref(W), int(on_dev), _stream_ptr(stream)),
               "moe_stack_load_layer")

    def forward(self, h_in, h_out=None, per_layer_out=None, stream=None):
        """h_in: fp16 CUDA [T, H]; per_layer_out: None or fp16 CUDA [n_layers, T, H] (receives every h_{l+1})."""
        import torch
        assert h_in.dtype == torch.float16 and h_in.is_cuda and h_in.is_contiguous()
        if h_out is None:
            h_out = torch.empty_like(h_in)
        if per_layer_out is not None:
            assert per_layer_out.dtype == torch.float16 and per_layer_out.is_contiguous()
            assert tuple(per_layer_out.shape) == (self.n_layers, *h_in.shape)
        _check(self.lib.moe_stack_forward(self.h, _ptr(h_in), _ptr(h_out), h_in.shape[0], _ptr(per_layer_out),
                                          _stream_ptr(stream)), "moe_stack_forward")
        return h_out

    def status(self):
        f = ctypes.c_uint32(0)
        s = self.lib.moe_stack_get_status(self.h, ctypes.byref(f))
        return s, f.value

    def layer_routing(self, layer, T):
        """The routing record of one layer's last call (the block test hook on the stack's own handle)."""
        import torch
        K = self.cfg.top_k
        hb = self.lib.moe_stack_layer(self.h, int(layer))
        ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
        w = torch.empty((T, K), dtype=torch.float32, device="cuda")
        _check(self.lib.moe_block_debug_last_routing(ctypes.c_void_p(hb), T, None, _ptr(ids), _ptr(w), None,
                                                     _stream_ptr(None)), "moe_block_debug_last_routing")
        return {"ids": ids, "w": w}


def upload_weights(w: dict, device="cuda"):
    """Canonical numpy arrays -> contiguous torch tensors on the device (fp16 arrays as uint16 bit patterns)."""
    import torch
    out = {}
    for k, v in w.items():
        a = np.ascontiguousarray(v)
        if a.dtype == np.float16:
            a = a.view(np.int16)          # bit patterns; the library reads them as fp16
        elif a.dtype == np.uint8:
            pass
        out[k] = torch.from_numpy(a).to(device)
    return out
