"""ctypes binding of libspecverify with the same entry-point names as the C ABI.

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (torch provides device memory and streams):

* ``wq``      int32 [N, K*bits/32]  (uint32 words reinterpreted)
* ``scales``  float16 [N, K/64],  ``biases`` float16 [N, K/64]
* activations bfloat16, logits / probabilities float32, tokens int32

Each call raises ``SVError`` when the library returns a non-OK status.  There
is no fallback: if the shared library is missing or the tensors are not on a
CUDA device the call fails.
"""

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "specverify.h")

SV_OK, SV_EINVAL, SV_EUNSUPPORTED, SV_ECUDA, SV_ETIMEOUT = range(5)

_c_void_p, _c_int, _c_size_t, _c_float, _c_u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t,
                                                  ctypes.c_float, ctypes.c_uint64)
_c_uint_p = ctypes.POINTER(ctypes.c_uint)
_c_i32_p = ctypes.POINTER(ctypes.c_int32)

class QWeight(ctypes.Structure):
    _fields_ = [("wq", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("N", ctypes.c_int), ("K", ctypes.c_int), ("packed", ctypes.c_void_p)]


class Layer(ctypes.Structure):
    _fields_ = [("qkv", QWeight), ("o", QWeight), ("gate_up", QWeight), ("down", QWeight)]


class Model(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("q_dim", ctypes.c_int),
                ("inter", ctypes.c_int), ("vocab", ctypes.c_int), ("bits", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("layers", ctypes.POINTER(Layer)), ("lm_head", QWeight)]


_c_model_p = ctypes.POINTER(Model)

SV_CAP_MAX = 31


class CapState(ctypes.Structure):
    """sv_cap_controller (host memory)."""
    _fields_ = [("max_cap", ctypes.c_int), ("verify_us", ctypes.c_double * (SV_CAP_MAX + 1)),
                ("draft_us", ctypes.c_double * (SV_CAP_MAX + 1)), ("overhead_us", ctypes.c_double),
                ("alpha", ctypes.c_double), ("probe_every", ctypes.c_int), ("probe_cap", ctypes.c_int),
                ("S", ctypes.c_double), ("F", ctypes.c_double), ("parked", ctypes.c_int),
                ("since_probe", ctypes.c_int)]


_c_cap_p = ctypes.POINTER(CapState)
_c_f64_p = ctypes.POINTER(ctypes.c_double)
_c_int_p = ctypes.POINTER(ctypes.c_int)

_SIGNATURES = {
    "sv_status_string": (ctypes.c_char_p, [_c_int]),
    "sv_last_error": (ctypes.c_char_p, []),
    "sv_version": (_c_int, []),
    "sv_device_error": (_c_int, [_c_uint_p]),
    "sv_selftest_bounded_wait": (_c_int, [ctypes.c_uint, _c_void_p]),
    "sv_qmm_workspace_bytes": (_c_size_t, [_c_int, _c_int, _c_int, _c_int]),
    "sv_qmm_verify": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p, _c_int,
                               _c_int, _c_void_p, _c_int, _c_void_p, _c_int, _c_void_p, _c_size_t, _c_void_p]),
    "sv_qmm_noalloc_scratch_bytes": (_c_size_t, []),
    "sv_qmm_verify_noalloc": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p,
                                       _c_int, _c_int, _c_void_p, _c_int, _c_void_p, _c_int, _c_void_p]),
    "sv_qmm_prepare": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_void_p, _c_int, _c_void_p,
                                _c_float, _c_void_p, _c_size_t, _c_void_p]),
    "sv_qmm_run": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_void_p,
                            _c_int, _c_void_p, _c_int, _c_void_p, _c_size_t, _c_void_p]),
    "sv_lm_head_workspace_bytes": (_c_size_t, [_c_int, _c_int, _c_int, _c_int]),
    "sv_lm_head_run": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                _c_void_p, _c_int, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_size_t,
                                _c_void_p]),
    "sv_round_workspace_bytes": (_c_size_t, [_c_model_p, _c_int]),
    "sv_qmm_pack_bytes": (_c_size_t, [_c_int, _c_int, _c_int]),
    "sv_qmm_pack": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p, _c_size_t,
                             _c_void_p]),
    "sv_round_plan_bytes": (_c_size_t, [_c_model_p]),
    "sv_round_plan_init": (_c_int, [_c_model_p, _c_void_p, _c_size_t]),
    "sv_verify_round": (_c_int, [_c_model_p, _c_void_p, _c_int, _c_i32_p, _c_void_p, _c_int, _c_float, _c_void_p, _c_int,
                                 _c_void_p, _c_void_p, _c_void_p, _c_int, _c_void_p, _c_void_p, _c_void_p,
                                 _c_size_t, _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "sv_lm_head_verify": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p,
                                   _c_int, _c_int, _c_float, _c_void_p, _c_int, _c_void_p, _c_void_p, _c_void_p,
                                   _c_void_p, _c_size_t, _c_void_p]),
    "sv_accept_workspace_bytes": (_c_size_t, [_c_int, _c_int]),
    "sv_spec_accept": (_c_int, [_c_void_p, _c_int, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_void_p,
                                _c_int, _c_int, _c_float, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_size_t,
                                _c_void_p]),
    "sv_spec_accept_batched": (_c_int, [_c_int, _c_i32_p, _c_void_p, _c_int, _c_void_p, _c_void_p, _c_void_p,
                                        _c_void_p, _c_int, _c_void_p, _c_int, _c_float, _c_void_p, _c_void_p,
                                        _c_void_p, _c_void_p, _c_size_t, _c_void_p]),
    "sv_philox_uniforms": (_c_int, [_c_u64, _c_u64, _c_u64, _c_int, _c_void_p, _c_void_p]),
    "sv_rmsnorm": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_void_p, _c_float, _c_void_p, _c_int, _c_void_p]),
    "sv_residual_add": (_c_int, [_c_void_p, _c_int, _c_void_p, _c_int, _c_int, _c_int, _c_void_p]),
    "sv_swiglu": (_c_int, [_c_void_p, _c_int, _c_void_p, _c_int, _c_int, _c_int, _c_void_p, _c_int, _c_void_p]),
    "sv_spec_accept_truncated": (_c_int, [_c_int, _c_i32_p, _c_void_p, _c_int, _c_void_p, _c_void_p, _c_void_p,
                                          _c_void_p, _c_int, _c_void_p, _c_int, _c_float, _c_void_p, _c_int,
                                          _c_float, _c_void_p, _c_void_p, _c_void_p, _c_size_t, _c_void_p]),
    "sv_truncate_probs": (_c_int, [_c_void_p, _c_int, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_float,
                                   _c_void_p]),
    "sv_logprobs": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_float, _c_void_p, _c_int, _c_void_p, _c_void_p,
                             _c_void_p, _c_void_p]),
    "sv_gather_qmm_workspace_bytes": (_c_size_t, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "sv_gather_qmm": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_void_p,
                               _c_int, _c_int, _c_void_p, _c_void_p, _c_int, _c_void_p, _c_int, _c_void_p,
                               _c_size_t, _c_void_p]),
    "sv_expected_committed": (ctypes.c_double, [ctypes.c_double, _c_int]),
    "sv_best_cap": (_c_int, [ctypes.c_double, _c_int, _c_f64_p, _c_f64_p, ctypes.c_double, _c_int_p, _c_f64_p]),
    "sv_verify_knee": (_c_int, [_c_f64_p, _c_int, ctypes.c_double, _c_int_p]),
    "sv_cap_init": (_c_int, [_c_cap_p, _c_int, _c_f64_p, _c_f64_p, ctypes.c_double, ctypes.c_double, _c_int, _c_int,
                             ctypes.c_double]),
    "sv_cap_next": (_c_int, [_c_cap_p, _c_int_p]),
    "sv_cap_update": (_c_int, [_c_cap_p, _c_int, _c_int]),
    "sv_cap_acceptance": (ctypes.c_double, [_c_cap_p]),
}


def _f64_array(values):
    arr = (ctypes.c_double * len(values))(*[float(v) for v in values])
    return ctypes.cast(arr, _c_f64_p), arr


class CapController:
    """sv_cap_controller: per-round draft cap from measured costs (host only)."""

    def __init__(self, lib, max_cap, verify_us, draft_us, overhead_us, alpha, probe_every, probe_cap, p0):
        self.lib, self.state = lib, CapState()
        v, self._v = _f64_array(verify_us)
        d, self._d = _f64_array(draft_us)
        _check(lib, lib.sv_cap_init(ctypes.byref(self.state), max_cap, v, d, overhead_us, alpha, probe_every,
                                    probe_cap, p0))

    def next_cap(self):
        c = ctypes.c_int()
        _check(self.lib, self.lib.sv_cap_next(ctypes.byref(self.state), ctypes.byref(c)))
        return c.value

    def update(self, cap, accepted):
        _check(self.lib, self.lib.sv_cap_update(ctypes.byref(self.state), cap, accepted))

    def p(self):
        return self.lib.sv_cap_acceptance(ctypes.byref(self.state))

    @property
    def parked(self):
        return bool(self.state.parked)


def best_cap(lib, p, verify_us, draft_us, overhead_us):
    """(cap, rate) from sv_best_cap; max_cap = len(verify_us) - 1."""
    v, _v = _f64_array(verify_us)
    d, _d = _f64_array(draft_us)
    c, r = ctypes.c_int(), ctypes.c_double()
    _check(lib, lib.sv_best_cap(p, len(verify_us) - 1, v, d, overhead_us, ctypes.byref(c), ctypes.byref(r)))
    return c.value, r.value


def verify_knee(lib, verify_us, tol):
    v, _v = _f64_array(verify_us)
    w = ctypes.c_int()
    _check(lib, lib.sv_verify_knee(v, len(verify_us), tol, ctypes.byref(w)))
    return w.value


def _check(lib, status):
    if status != SV_OK:
        raise SVError(status, lib.sv_last_error().decode())


class SVError(RuntimeError):
    def __init__(self, status, detail):
        super().__init__("%s (status %d): %s" % (_STATUS_NAMES.get(status, "?"), status, detail))
        self.status = status


_STATUS_NAMES = {0: "SV_OK", 1: "SV_EINVAL", 2: "SV_EUNSUPPORTED", 3: "SV_ECUDA", 4: "SV_ETIMEOUT"}


def header_functions():
    """Names of the functions declared in include/specverify.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(sv_\w+)\s*\(", text, flags=re.M)))


def load_library(path=LIB_PATH):
    """dlopen the library and attach the argument types (no device work)."""
    if not os.path.exists(path):
        raise RuntimeError("libspecverify.so is not built (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Library:
    """The loaded library plus tensor-level helpers named after the C calls."""

    def __init__(self, path=LIB_PATH):
        self.lib = load_library(path)

    # -------------------------------------------------------------- plumbing
    def check(self, status):
        if status != SV_OK:
            raise SVError(status, self.lib.sv_last_error().decode())

    def device_error(self):
        bits = ctypes.c_uint(0)
        st = self.lib.sv_device_error(ctypes.byref(bits))
        if st not in (SV_OK, SV_ETIMEOUT):
            self.check(st)
        return bits.value

    @staticmethod
    def workspace(nbytes, device="cuda"):
        """A zero-filled, 256-byte aligned device buffer (torch allocates it)."""
        import torch
        return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)

    # ------------------------------------------------------------------ qmm
    def qmm_workspace_bytes(self, M, N, K, bits):
        return self.lib.sv_qmm_workspace_bytes(M, N, K, bits)

    def qmm_verify(self, wq, scales, biases, K, bits, x, y=None, residual=None, workspace=None, stream=None):
        import torch
        M, N = x.shape[0], wq.shape[0]
        if y is None:
            y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
        if workspace is None:
            workspace = self.workspace(self.qmm_workspace_bytes(M, N, K, bits), x.device)
        self.check(self.lib.sv_qmm_verify(
            _ptr(wq), _ptr(scales), _ptr(biases), N, K, bits, 64, _ptr(x), x.stride(0), M, _ptr(y), y.stride(0),
            _ptr(residual), residual.stride(0) if residual is not None else 0, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
        return y

    def qmm_verify_noalloc(self, wq, scales, biases, K, bits, x, y=None, residual=None, stream=None):
        """sv_qmm_verify without a workspace (scratch in the library's own device array)."""
        import torch
        M, N = x.shape[0], wq.shape[0]
        if y is None:
            y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
        self.check(self.lib.sv_qmm_verify_noalloc(
            _ptr(wq), _ptr(scales), _ptr(biases), N, K, bits, 64, _ptr(x), x.stride(0), M, _ptr(y), y.stride(0),
            _ptr(residual), residual.stride(0) if residual is not None else 0, _stream(stream)))
        return y

    def qmm_prepare(self, x, K, bits, mode=0, x2=None, rms_weight=None, eps=1e-6, workspace=None, stream=None):
        M = x.shape[0]
        self.check(self.lib.sv_qmm_prepare(
            _ptr(x), x.stride(0), M, K, bits, mode, _ptr(x2), x2.stride(0) if x2 is not None else 0,
            _ptr(rms_weight), eps, _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))

    def qmm_run(self, wq, scales, biases, K, bits, M, y=None, residual=None, workspace=None, stream=None):
        import torch
        N = wq.shape[0]
        if y is None:
            y = torch.empty((M, N), dtype=torch.bfloat16, device=wq.device)
        self.check(self.lib.sv_qmm_run(
            _ptr(wq), _ptr(scales), _ptr(biases), N, K, bits, 64, M, _ptr(y), y.stride(0), _ptr(residual),
            residual.stride(0) if residual is not None else 0, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
        return y

    # -------------------------------------------------------------- lm_head
    def lm_head_workspace_bytes(self, M, V, K, bits):
        return self.lib.sv_lm_head_workspace_bytes(M, V, K, bits)

    def lm_head_verify(self, wq, scales, biases, K, bits, x, temperature, logits=None, stats=True, workspace=None,
                       stream=None):
        import torch
        M, V = x.shape[0], wq.shape[0]
        dev = x.device
        if logits is None:
            logits = torch.empty((M, V), dtype=torch.float32, device=dev)
        row_max = row_sumexp = row_argmax = None
        if stats:
            row_max = torch.empty(M, dtype=torch.float32, device=dev)
            row_sumexp = torch.zeros(M, dtype=torch.float32, device=dev)
            row_argmax = torch.empty(M, dtype=torch.int32, device=dev)
        if workspace is None:
            workspace = self.workspace(self.lm_head_workspace_bytes(M, V, K, bits), dev)
        self.check(self.lib.sv_lm_head_verify(
            _ptr(wq), _ptr(scales), _ptr(biases), V, K, bits, 64, _ptr(x), x.stride(0), M, float(temperature),
            _ptr(logits), logits.stride(0), _ptr(row_max), _ptr(row_sumexp), _ptr(row_argmax), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
        return logits, row_max, row_sumexp, row_argmax

    def lm_head_run(self, wq, scales, biases, K, bits, M, temperature, logits=None, stats=None, workspace=None,
                    stream=None):
        import torch
        V = wq.shape[0]
        if logits is None:
            logits = torch.empty((M, V), dtype=torch.float32, device=wq.device)
        rmax, rsum, rarg = stats if stats is not None else (None, None, None)
        self.check(self.lib.sv_lm_head_run(
            _ptr(wq), _ptr(scales), _ptr(biases), V, K, bits, 64, M, float(temperature), _ptr(logits),
            logits.stride(0), _ptr(rmax), _ptr(rsum), _ptr(rarg), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
        return logits

    # ---------------------------------------------------------------- round
    def make_model(self, layers, lm_head, hidden, q_dim, inter, vocab, bits, rms_eps=1e-6):
        """A ctypes sv_model over device weight dicts {'wq','scales','biases'}, with its round plan
        (``model.plan``, a device tensor built by sv_round_plan_init).

        ``layers``: list of dicts with keys qkv, o, gate_up, down."""
        def qw(w):
            packed = w.get("packed")
            return QWeight(w["wq"].data_ptr(), w["scales"].data_ptr(), w["biases"].data_ptr(), w["wq"].shape[0],
                           w["K"], packed.data_ptr() if packed is not None else None)
        arr = (Layer * len(layers))(*[Layer(qw(l["qkv"]), qw(l["o"]), qw(l["gate_up"]), qw(l["down"]))
                                      for l in layers])
        m = Model(len(layers), hidden, q_dim, inter, vocab, bits, rms_eps, arr, qw(lm_head))
        # the struct holds raw device pointers: keep the tensors (and the array) alive with it
        m._keep = (arr, layers, lm_head)
        nbytes = self.lib.sv_round_plan_bytes(ctypes.byref(m))
        if nbytes == 0:
            raise SVError(SV_EINVAL, "sv_round_plan_bytes: model rejected")
        m.plan = self.workspace(nbytes, device=lm_head["wq"].device)
        self.check(self.lib.sv_round_plan_init(ctypes.byref(m), _ptr(m.plan), nbytes))
        return m

    def pack(self, w, stream=None):
        """Unit-packed copy of a device weight dict (sv_qmm_pack); returns a uint8 device tensor."""
        import torch
        N, K, bits = w["wq"].shape[0], w["K"], w["bits"]
        nbytes = self.lib.sv_qmm_pack_bytes(N, K, bits)
        if nbytes == 0:
            raise SVError(SV_EUNSUPPORTED, "sv_qmm_pack_bytes: unsupported shape")
        out = torch.empty(nbytes, dtype=torch.uint8, device=w["wq"].device)
        self.check(self.lib.sv_qmm_pack(_ptr(w["wq"]), _ptr(w["scales"]), _ptr(w["biases"]), N, K, bits, 64, _ptr(out),
                                        nbytes, _stream(stream)))
        return out

    def round_workspace_bytes(self, model, rows):
        return self.lib.sv_round_workspace_bytes(ctypes.byref(model), rows)

    def verify_round(self, model, row_offsets, hidden, temperature, logits, out_len, out_tokens, workspace,
                     q=None, draft=None, u=None, stream=None, events=None, accept_wait=None):
        """events: optional (start, stop) torch.cuda.Event pair recorded around the matmul launch;
        accept_wait: optional torch.cuda.Event the accept step waits for (q, draft and u copied in
        on another stream while the projections run)."""
        B = len(row_offsets) - 1
        offs = (ctypes.c_int32 * (B + 1))(*[int(v) for v in row_offsets])
        ev0 = ev1 = None
        if events is not None:
            ev0, ev1 = (ctypes.c_void_p(e.cuda_event) for e in events)
        self.check(self.lib.sv_verify_round(
            ctypes.byref(model), _ptr(model.plan), B, offs, _ptr(hidden), hidden.stride(0), float(temperature), _ptr(q),
            q.stride(0) if q is not None else 0, _ptr(draft), _ptr(u), _ptr(logits), logits.stride(0),
            _ptr(out_len), _ptr(out_tokens), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream), ev0, ev1, ctypes.c_void_p(accept_wait.cuda_event) if accept_wait is not None else None))

    # --------------------------------------------------------------- accept
    def accept_workspace_bytes(self, B, rows):
        return self.lib.sv_accept_workspace_bytes(B, rows)

    def spec_accept(self, logits, draft, temperature, q=None, u=None, stats=None, workspace=None, stream=None):
        """stats: (row_max, row_sumexp, row_argmax) from lm_head_verify, or None."""
        import torch
        m = logits.shape[0] - 1
        V = logits.shape[1]
        dev = logits.device
        out_len = torch.zeros(1, dtype=torch.int32, device=dev)
        out_tokens = torch.full((m + 1,), -1, dtype=torch.int32, device=dev)
        if workspace is None:
            workspace = self.workspace(self.accept_workspace_bytes(1, m + 1), dev)
        rmax, rsum, rarg = stats if stats is not None else (None, None, None)
        self.check(self.lib.sv_spec_accept(
            _ptr(logits), logits.stride(0), _ptr(rmax), _ptr(rsum), _ptr(rarg), _ptr(q),
            q.stride(0) if q is not None else 0, _ptr(draft), m, V, float(temperature), _ptr(u), _ptr(out_len),
            _ptr(out_tokens), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
        return out_len, out_tokens

    def spec_accept_batched(self, row_offsets, logits, drafts, temperature, q=None, u=None, stats=None,
                            workspace=None, stream=None):
        import torch
        B = len(row_offsets) - 1
        rows = int(row_offsets[-1])
        V = logits.shape[1]
        dev = logits.device
        offs = (ctypes.c_int32 * (B + 1))(*[int(v) for v in row_offsets])
        out_len = torch.zeros(B, dtype=torch.int32, device=dev)
        out_tokens = torch.full((rows,), -1, dtype=torch.int32, device=dev)
        if workspace is None:
            workspace = self.workspace(self.accept_workspace_bytes(B, rows), dev)
        rmax, rsum, rarg = stats if stats is not None else (None, None, None)
        self.check(self.lib.sv_spec_accept_batched(
            B, offs, _ptr(logits), logits.stride(0), _ptr(rmax), _ptr(rsum), _ptr(rarg), _ptr(q),
            q.stride(0) if q is not None else 0, _ptr(drafts), V, float(temperature), _ptr(u), _ptr(out_len),
            _ptr(out_tokens), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
        return out_len, out_tokens

    def spec_accept_truncated(self, row_offsets, logits, drafts, temperature, top_k, top_p, q=None, u=None,
                              stats=None, workspace=None, stream=None):
        import torch
        B = len(row_offsets) - 1
        rows = int(row_offsets[-1])
        V = logits.shape[1]
        dev = logits.device
        offs = (ctypes.c_int32 * (B + 1))(*[int(v) for v in row_offsets])
        out_len = torch.zeros(B, dtype=torch.int32, device=dev)
        out_tokens = torch.full((rows,), -1, dtype=torch.int32, device=dev)
        if workspace is None:
            workspace = self.workspace(self.accept_workspace_bytes(B, rows), dev)
        rmax, rsum, rarg = stats if stats is not None else (None, None, None)
        self.check(self.lib.sv_spec_accept_truncated(
            B, offs, _ptr(logits), logits.stride(0), _ptr(rmax), _ptr(rsum), _ptr(rarg), _ptr(q),
            q.stride(0) if q is not None else 0, _ptr(drafts), V, float(temperature), _ptr(u), int(top_k),
            float(top_p), _ptr(out_len), _ptr(out_tokens), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
        return out_len, out_tokens

    def truncate_probs(self, probs, top_k, top_p, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(probs)
        self.check(self.lib.sv_truncate_probs(_ptr(probs), probs.stride(0), _ptr(out), out.stride(0), probs.shape[0],
                                              probs.shape[1], int(top_k), float(top_p), _stream(stream)))
        return out

    def logprobs(self, logits, temperature, chosen=None, top_n=0, stream=None):
        """(chosen_logprob [rows] or None, top_ids [rows, top_n], top_logprobs [rows, top_n])."""
        import torch
        rows, V = logits.shape
        dev = logits.device
        clp = torch.empty(rows, dtype=torch.float32, device=dev) if chosen is not None else None
        ids = torch.empty((rows, top_n), dtype=torch.int32, device=dev)
        tlp = torch.empty((rows, top_n), dtype=torch.float32, device=dev)
        self.check(self.lib.sv_logprobs(_ptr(logits), logits.stride(0), rows, V, float(temperature), _ptr(chosen),
                                        int(top_n), _ptr(clp), _ptr(ids) if top_n else None,
                                        _ptr(tlp) if top_n else None, _stream(stream)))
        return clp, ids, tlp

    # --------------------------------------------------------------- gather
    def gather_qmm(self, wq, scales, biases, E, K, bits, x, pair_rows, pair_experts, y=None, workspace=None,
                   stream=None):
        """Stacked expert weights [E*N, ...]; pair_rows / pair_experts int32 device tensors [P]."""
        import torch
        N = wq.shape[0] // E
        M, P = x.shape[0], pair_rows.shape[0]
        if y is None:
            y = torch.empty((P, N), dtype=torch.bfloat16, device=x.device)
        if workspace is None:
            nbytes = self.lib.sv_gather_qmm_workspace_bytes(P, M, N, K, E, bits)
            if nbytes == 0:
                raise SVError(SV_EINVAL, "sv_gather_qmm_workspace_bytes: unsupported sizes")
            workspace = self.workspace(nbytes, x.device)
        self.check(self.lib.sv_gather_qmm(_ptr(wq), _ptr(scales), _ptr(biases), E, N, K, bits, 64, _ptr(x),
                                          x.stride(0), M, _ptr(pair_rows), _ptr(pair_experts), P, _ptr(y), y.stride(0),
                                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream)))
        return y

    # --------------------------------------------------------------- philox
    def philox_uniforms(self, seed, subsequence, offset, n, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(n, dtype=torch.float32, device="cuda")
        self.check(self.lib.sv_philox_uniforms(seed, subsequence, offset, n, _ptr(out), _stream(stream)))
        return out

    # ----------------------------------------------------------------- glue
    def rmsnorm(self, x, weight=None, eps=1e-6, y=None, stream=None):
        import torch
        if y is None:
            y = torch.empty_like(x)
        self.check(self.lib.sv_rmsnorm(_ptr(x), x.stride(0), x.shape[0], x.shape[1], _ptr(weight), eps, _ptr(y),
                                       y.stride(0), _stream(stream)))
        return y

    def residual_add(self, h, t, stream=None):
        self.check(self.lib.sv_residual_add(_ptr(h), h.stride(0), _ptr(t), t.stride(0), h.shape[0], h.shape[1],
                                            _stream(stream)))
        return h

    def swiglu(self, g, u, s=None, stream=None):
        import torch
        if s is None:
            s = torch.empty_like(g)
        self.check(self.lib.sv_swiglu(_ptr(g), g.stride(0), _ptr(u), u.stride(0), g.shape[0], g.shape[1], _ptr(s),
                                      s.stride(0), _stream(stream)))
        return s


_LIB = None


def load():
    """The process-wide Library; builds nothing and falls back to nothing."""
    global _LIB
    if _LIB is None:
        _LIB = Library()
    return _LIB
