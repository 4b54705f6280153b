"""ctypes binding of ``libkvpool.so`` (argument marshalling only).

Every step of the path runs in the library's CUDA kernels; this module only
turns torch tensors into device pointers and the current torch stream into a
``cudaStream_t``. There is no fallback: if the library is missing or the
device is not an sm_103 GPU the calls raise.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvpool.so")

OK = 0
ERRORS = {
    -1: "INVALID_ARG", -2: "STATE", -3: "CUDA", -4: "OOM", -5: "NONFINITE", -6: "TIMEOUT",
    -7: "UNSUPPORTED",
}


class KVPoolError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({_lib().kvpool_strerror(code).decode()})")


class Tail(ctypes.Structure):
    _fields_ = [("K", ctypes.c_void_p), ("V", ctypes.c_void_p), ("len", ctypes.c_void_p),
                ("T_max", ctypes.c_int)]


class LayerView(ctypes.Structure):
    _fields_ = [("kq", ctypes.c_void_p), ("vcodes", ctypes.c_void_p), ("vnorm", ctypes.c_void_p),
                ("kscale", ctypes.c_void_p), ("ctx", ctypes.c_int), ("ctx_padded", ctypes.c_int),
                ("bits", ctypes.c_int), ("compressed", ctypes.c_int),
                ("kscales", ctypes.c_void_p), ("k_block", ctypes.c_int), ("len", ctypes.c_int),
                ("group_bits", ctypes.c_void_p), ("group_off", ctypes.c_void_p), ("mixed", ctypes.c_int)]


_LIB = None

# name -> (restype, argtypes); the C declarations are in include/kvpool.h
_SIGS = {
    "kvpool_create": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]),
    "kvpool_create_ex": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_int]),
    "kvpool_export_kscales": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "kvpool_append": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int, ctypes.c_void_p]),
    "kvpool_append_bits": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "kvpool_layer_widths": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]),
    "kvpool_layer_len": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "kvpool_sensitivity": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]),
    "kvpool_allocate_bits": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_void_p]),
    "kvpool_destroy": (None, [ctypes.c_void_p]),
    "kvpool_compress": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "kvpool_attend": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_float, ctypes.c_void_p]),
    "kvpool_decompress": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p]),
    "kvpool_compress_layers": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "kvpool_decompress_layers": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "kvpool_pool_bytes": (ctypes.c_size_t, [ctypes.c_void_p]),
    "kvpool_device_bytes": (ctypes.c_size_t, [ctypes.c_void_p]),
    "kvpool_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "kvpool_reset_layer": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "kvpool_layer_view": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(LayerView)]),
    "kvpool_codebook": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "kvpool_export_layer": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5),
    "kvpool_import_layer": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5),
    "kvpool_import_layer_blocks": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int] + [ctypes.c_void_p] * 5 +
                                   [ctypes.c_int, ctypes.c_void_p]),
    "kvpool_attend_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 +
                              [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p]),
    "kvpool_attend_ws": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "kvpool_attend_ws_bytes": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]),
    "kvpool_attend_partial": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p]),
    "kvpool_merge_partials": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                             ctypes.c_void_p]),
    "kvpool_strerror": (ctypes.c_char_p, [ctypes.c_int]),
}


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m shared_quantized_kv_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def lib():
    """The loaded library (ctypes.CDLL)."""
    return _lib()


def _check(rc: int, what: str):
    if rc != OK:
        raise KVPoolError(rc, what)


def _stream_ptr(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev_ptr(t, dtype, name):
    import torch

    if t is None:
        return None
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")
    return ctypes.c_void_p(t.data_ptr())


def codebook(bits: int):
    """The library's float32 (centroids, midpoints) for ``bits`` (host)."""
    import numpy as np

    c = np.zeros(1 << bits, np.float32)
    m = np.zeros((1 << bits) - 1, np.float32)
    _check(_lib().kvpool_codebook(bits, c.ctypes.data, m.ctypes.data), "kvpool_codebook")
    return c, m


def sensitivity(Q, recent, kv_heads, softmax_scale=0.0, stream=None):
    """A layer's local attention-error estimate s (float) and the per-row
    values r (float32 [agents * q_heads], device) from recent tokens: Q bf16
    [agents, q_heads, d]; recent = (K, V, lens) with K, V bf16 [agents,
    kv_heads, T_max, d] and lens int32 [agents] (device)."""
    import torch

    A, Hq, d = Q.shape
    K, V, lens = recent
    t = Tail(_dev_ptr(K, torch.bfloat16, "recent K").value, _dev_ptr(V, torch.bfloat16, "recent V").value,
             _dev_ptr(lens, torch.int32, "recent len").value, K.shape[2])
    rows = torch.empty(A * Hq, dtype=torch.float32, device=Q.device)
    score = torch.empty(1, dtype=torch.float32, device=Q.device)
    _check(_lib().kvpool_sensitivity(_dev_ptr(Q, torch.bfloat16, "Q"), A, Hq, ctypes.byref(t), kv_heads, d,
                                     softmax_scale, rows.data_ptr(), score.data_ptr(), _stream_ptr(stream)),
           "kvpool_sensitivity")
    return float(score.cpu()[0]), rows


def merge_partials(ml, acc, Q, kv_heads, tail=None, out=None, softmax_scale=0.0, stream=None):
    """kvpool_merge_partials: ml float32 [parts, kv_heads, rows, 2] and acc
    float32 [parts, kv_heads, rows, d] from attend_partial (device); Q bf16
    [agents, q_heads, d]; tail None or (K, V, lens) as for attend. Returns out
    float32 [agents, q_heads, d]."""
    import torch

    A, Hq, d = Q.shape
    parts = ml.shape[0]
    if out is None:
        out = torch.empty((A, Hq, d), dtype=torch.float32, device=Q.device)
    tp = None
    if tail is not None:
        Kt, Vt, lens = tail
        t = Tail(_dev_ptr(Kt, torch.bfloat16, "tail K").value, _dev_ptr(Vt, torch.bfloat16, "tail V").value,
                 _dev_ptr(lens, torch.int32, "tail len").value, Kt.shape[2])
        tp = ctypes.byref(t)
    _check(_lib().kvpool_merge_partials(parts, _dev_ptr(ml, torch.float32, "ml"), _dev_ptr(acc, torch.float32, "acc"),
                                        kv_heads, d, _dev_ptr(Q, torch.bfloat16, "Q"), A, Hq, tp,
                                        _dev_ptr(out, torch.float32, "out"), softmax_scale, _stream_ptr(stream)),
           "kvpool_merge_partials")
    return out


def allocate_bits(sens, cost, budget):
    """Per-layer V widths (list of 2, 3, 4) minimising sum D_b s^2 within
    sum cost * bits <= budget (host only)."""
    import numpy as np

    L = len(sens)
    s = np.ascontiguousarray(sens, dtype=np.float64)
    c = np.ascontiguousarray(cost, dtype=np.int64)
    out = np.zeros(L, dtype=np.uint8)
    _check(_lib().kvpool_allocate_bits(L, s.ctypes.data, c.ctypes.data, int(budget), out.ctypes.data),
           "kvpool_allocate_bits")
    return [int(b) for b in out]


class KVPool:
    """One shared pool (a ``kvpool_t``) on the current CUDA device."""

    def __init__(self, layers, kv_heads, head_dim, ctx, bits=None, max_rows=0, k_block=0):
        """k_block: 0 (one K scale per layer) or 32 (one per 32 elements)."""
        self.layers, self.kv_heads, self.head_dim, self.ctx = layers, kv_heads, head_dim, ctx
        self.bits = list(bits) if bits is not None else [3] * layers
        self.k_block = k_block
        arr = (ctypes.c_uint8 * layers)(*self.bits)
        h = ctypes.c_void_p()
        _check(_lib().kvpool_create_ex(ctypes.byref(h), layers, kv_heads, head_dim, ctx,
                                       ctypes.cast(arr, ctypes.c_void_p), max_rows, k_block),
               "kvpool_create_ex")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            _lib().kvpool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def compress(self, layer, K, V, stream=None):
        import torch

        _check(_lib().kvpool_compress(self._h, layer, _dev_ptr(K, torch.bfloat16, "K"),
                                      _dev_ptr(V, torch.bfloat16, "V"), _stream_ptr(stream)),
               "kvpool_compress")

    def compress_layers(self, layers, Ks, Vs, stream=None):
        """compress() of every layer in ``layers`` (K = Ks[i], V = Vs[i]) in
        one call: one max|K| kernel for all of them, one encode kernel per V
        width among them."""
        import torch

        n = len(layers)
        if len(Ks) != n or len(Vs) != n:
            raise ValueError("layers, Ks and Vs must have the same length")
        lay = (ctypes.c_int * max(n, 1))(*[int(l) for l in layers])
        kp = (ctypes.c_void_p * max(n, 1))(*[_dev_ptr(K, torch.bfloat16, "K").value for K in Ks])
        vp = (ctypes.c_void_p * max(n, 1))(*[_dev_ptr(V, torch.bfloat16, "V").value for V in Vs])
        _check(_lib().kvpool_compress_layers(self._h, n, lay, kp, vp, _stream_ptr(stream)),
               "kvpool_compress_layers")

    def append(self, layer, K, V, bits=None, stream=None):
        """Append tokens to a block-scaled layer: K, V bf16 [kv_heads, n, d]
        (device) become tokens [len, len + n) of the layer, their V codes at
        `bits` (None: the layer's width; else 2..that width)."""
        import torch

        kp, vp = _dev_ptr(K, torch.bfloat16, "K"), _dev_ptr(V, torch.bfloat16, "V")
        if bits is None:
            _check(_lib().kvpool_append(self._h, layer, kp, vp, int(K.shape[1]), _stream_ptr(stream)),
                   "kvpool_append")
        else:
            _check(_lib().kvpool_append_bits(self._h, layer, kp, vp, int(K.shape[1]), int(bits),
                                             _stream_ptr(stream)), "kvpool_append_bits")

    def layer_widths(self, layer):
        """V width of every 32-token group the layer holds (list of int)."""
        n = int(_lib().kvpool_layer_widths(self._h, layer, None, 0))
        if n < 0:
            raise KVPoolError(n, "kvpool_layer_widths")
        buf = (ctypes.c_uint8 * max(n, 1))()
        _check(min(0, _lib().kvpool_layer_widths(self._h, layer, buf, n)), "kvpool_layer_widths")
        return [int(b) for b in buf[:n]]

    def layer_len(self, layer) -> int:
        """Tokens the layer holds (ctx once compressed)."""
        n = int(_lib().kvpool_layer_len(self._h, layer))
        if n < 0:
            raise KVPoolError(n, "kvpool_layer_len")
        return n

    def attend(self, layer, Q, out=None, tail=None, softmax_scale=0.0, stream=None):
        """Q: bf16 [agents, q_heads, d]; tail: None or (K, V, lens) with K, V
        bf16 [agents, kv_heads, T_max, d] and lens int32 [agents] (device).
        Returns out: float32 [agents, q_heads, d]."""
        import torch

        A, Hq, d = Q.shape
        if out is None:
            out = torch.empty((A, Hq, d), dtype=torch.float32, device=Q.device)
        tp = None
        if tail is not None:
            Kt, Vt, lens = tail
            self._tail = Tail(_dev_ptr(Kt, torch.bfloat16, "tail K").value,
                              _dev_ptr(Vt, torch.bfloat16, "tail V").value,
                              _dev_ptr(lens, torch.int32, "tail len").value, Kt.shape[2])
            tp = ctypes.byref(self._tail)
        _check(_lib().kvpool_attend(self._h, layer, _dev_ptr(Q, torch.bfloat16, "Q"), A, Hq, tp,
                                    _dev_ptr(out, torch.float32, "out"), softmax_scale,
                                    _stream_ptr(stream)), "kvpool_attend")
        return out

    def attend_ws_bytes(self, agents, q_heads) -> int:
        """Workspace bytes kvpool_attend_ws needs for this many agents."""
        return int(_lib().kvpool_attend_ws_bytes(self._h, int(agents), int(q_heads)))

    def attend_ws(self, layer, Q, workspace=None, out=None, tail=None, softmax_scale=0.0, stream=None):
        """kvpool_attend_ws: as attend, through a device workspace (uint8
        tensor of at least attend_ws_bytes bytes; allocated here if None)."""
        import torch

        A, Hq, d = Q.shape
        if out is None:
            out = torch.empty((A, Hq, d), dtype=torch.float32, device=Q.device)
        if workspace is None:
            workspace = torch.empty(max(self.attend_ws_bytes(A, Hq), 16), dtype=torch.uint8, device=Q.device)
        tp = None
        if tail is not None:
            Kt, Vt, lens = tail
            self._tail = Tail(_dev_ptr(Kt, torch.bfloat16, "tail K").value,
                              _dev_ptr(Vt, torch.bfloat16, "tail V").value,
                              _dev_ptr(lens, torch.int32, "tail len").value, Kt.shape[2])
            tp = ctypes.byref(self._tail)
        _check(_lib().kvpool_attend_ws(self._h, layer, _dev_ptr(Q, torch.bfloat16, "Q"), A, Hq, tp,
                                       _dev_ptr(out, torch.float32, "out"), softmax_scale,
                                       workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                       _stream_ptr(stream)), "kvpool_attend_ws")
        return out

    def attend_partial(self, layer, Q, t_begin, t_end, ml=None, acc=None, softmax_scale=0.0, stream=None):
        """kvpool_attend_partial over pool tokens [t_begin, t_end): returns
        (ml float32 [kv_heads, rows, 2], acc float32 [kv_heads, rows, d]),
        rows = agents * (q_heads / kv_heads)."""
        import torch

        A, Hq, d = Q.shape
        R = A * (Hq // self.kv_heads)
        if ml is None:
            ml = torch.empty((self.kv_heads, R, 2), dtype=torch.float32, device=Q.device)
        if acc is None:
            acc = torch.empty((self.kv_heads, R, d), dtype=torch.float32, device=Q.device)
        _check(_lib().kvpool_attend_partial(self._h, layer, _dev_ptr(Q, torch.bfloat16, "Q"), A, Hq, t_begin, t_end,
                                            _dev_ptr(ml, torch.float32, "ml"), _dev_ptr(acc, torch.float32, "acc"),
                                            softmax_scale, _stream_ptr(stream)), "kvpool_attend_partial")
        return ml, acc

    def decompress(self, layer, K_out=None, V_out=None, stream=None):
        import torch

        shape = (self.kv_heads, self.layer_len(layer), self.head_dim)
        dev = torch.device("cuda", torch.cuda.current_device())
        if K_out is None:
            K_out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        if V_out is None:
            V_out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        _check(_lib().kvpool_decompress(self._h, layer, _dev_ptr(K_out, torch.bfloat16, "K_out"),
                                        _dev_ptr(V_out, torch.bfloat16, "V_out"),
                                        _stream_ptr(stream)), "kvpool_decompress")
        return K_out, V_out

    def decompress_layers(self, layers, K_outs=None, V_outs=None, stream=None):
        """decompress() of every layer in ``layers`` in one launch per V
        width. K_outs / V_outs: lists of bf16 [kv_heads, len, d] tensors
        (allocated when None). Returns (K_outs, V_outs)."""
        import torch

        n = len(layers)
        dev = torch.device("cuda", torch.cuda.current_device())

        def outs(given):
            if given is not None:
                if len(given) != n:
                    raise ValueError("one output per layer")
                return list(given)
            return [torch.empty((self.kv_heads, self.layer_len(l), self.head_dim), dtype=torch.bfloat16,
                                device=dev) for l in layers]

        K_outs, V_outs = outs(K_outs), outs(V_outs)
        lay = (ctypes.c_int * max(n, 1))(*[int(l) for l in layers])
        kp = (ctypes.c_void_p * max(n, 1))(*[_dev_ptr(K, torch.bfloat16, "K_out").value for K in K_outs])
        vp = (ctypes.c_void_p * max(n, 1))(*[_dev_ptr(V, torch.bfloat16, "V_out").value for V in V_outs])
        _check(_lib().kvpool_decompress_layers(self._h, n, lay, kp, vp, _stream_ptr(stream)),
               "kvpool_decompress_layers")
        return K_outs, V_outs

    def pool_bytes(self) -> int:
        return int(_lib().kvpool_pool_bytes(self._h))

    def device_bytes(self) -> int:
        return int(_lib().kvpool_device_bytes(self._h))

    def status(self, stream=None) -> int:
        """Synchronise and return (and clear) the device status code."""
        return int(_lib().kvpool_status(self._h, _stream_ptr(stream)))

    def reset_layer(self, layer):
        _check(_lib().kvpool_reset_layer(self._h, layer), "kvpool_reset_layer")

    def layer_view(self, layer) -> LayerView:
        v = LayerView()
        _check(_lib().kvpool_layer_view(self._h, layer, ctypes.byref(v)), "kvpool_layer_view")
        return v

    def export_layer(self, layer, stream=None):
        """The layer's stored bytes as device tensors (token padding removed):
        kq int8 [Hk, ctx, d], vcodes uint8 [Hk, ceil(ctx/32), d, 4*bits] (per
        32-token group, one packed code sequence per coordinate; a layer of
        per-group widths: [Hk, sum_g d*4*b_g], its groups back to back),
        vnorm float32 [Hk, ctx], kscale float32 [1]."""
        import torch

        bits = self.bits[layer]
        dev = torch.device("cuda", torch.cuda.current_device())
        Hk, T, d = self.kv_heads, self.layer_len(layer), self.head_dim
        kq = torch.empty((Hk, T, d), dtype=torch.int8, device=dev)
        if self.layer_view(layer).mixed:
            vc = torch.empty((Hk, d * 4 * sum(self.layer_widths(layer))), dtype=torch.uint8, device=dev)
        else:
            vc = torch.empty((Hk, (T + 31) // 32, d, 4 * bits), dtype=torch.uint8, device=dev)
        vn = torch.empty((Hk, T), dtype=torch.float32, device=dev)
        ks = torch.empty(1, dtype=torch.float32, device=dev)
        _check(_lib().kvpool_export_layer(self._h, layer, kq.data_ptr(), vc.data_ptr(),
                                          vn.data_ptr(), ks.data_ptr(), _stream_ptr(stream)),
               "kvpool_export_layer")
        return kq, vc, vn, ks

    def import_layer(self, layer, kq, vcodes, vnorm, kscale, stream=None):
        _check(_lib().kvpool_import_layer(self._h, layer, kq.data_ptr(), vcodes.data_ptr(),
                                          vnorm.data_ptr(), kscale.data_ptr(),
                                          _stream_ptr(stream)), "kvpool_import_layer")

    def import_layer_blocks(self, layer, kq, vcodes, vnorm, kscales, widths=None, stream=None):
        """Load a block-scaled layer: kq int8 [Hk, len, d], vcodes uint8 (the
        layer's groups per head back to back), vnorm float32 [Hk, len],
        kscales float32 [Hk, len, d/32] (device tensors); widths: list of the
        groups' V widths (None: the layer's width)."""
        buf = None
        if widths is not None:
            buf = (ctypes.c_uint8 * max(len(widths), 1))(*widths)
        _check(_lib().kvpool_import_layer_blocks(self._h, layer, kq.data_ptr(), vcodes.data_ptr(), vnorm.data_ptr(),
                                                 kscales.data_ptr(), buf, int(kq.shape[1]), _stream_ptr(stream)),
               "kvpool_import_layer_blocks")

    def export_kscales(self, layer, stream=None):
        """Block scales of a block-scaled pool's layer: float32 [Hk, ctx, d/32]."""
        import torch

        out = torch.empty((self.kv_heads, self.layer_len(layer), self.head_dim // 32), dtype=torch.float32,
                          device="cuda")
        _check(_lib().kvpool_export_kscales(self._h, layer, out.data_ptr(), _stream_ptr(stream)),
               "kvpool_export_kscales")
        return out

    def read_layer(self, layer):
        """Host numpy copies of one layer's stored bytes (see export_layer)."""
        kq, vc, vn, ks = self.export_layer(layer)
        d = dict(kq=kq.cpu().numpy(), vcodes=vc.cpu().numpy(), vnorm=vn.cpu().numpy(),
                 kscale=ks.cpu().numpy()[0])
        if self.k_block:
            d["kscales"] = self.export_kscales(layer).cpu().numpy()
        return d
