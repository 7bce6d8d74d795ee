"""Thin ctypes binding of libblk (include/blk.h): argument marshalling only.

PyTorch provides device memory and streams; every step of the block runs in
the library's CUDA kernels. There is no fallback: if libblk.so is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_longlong, c_size_t, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libblk.so")

BLK_OK = 0
STATUS_NAMES = {0: "BLK_OK", 1: "BLK_ERR_INVALID_ARG", 2: "BLK_ERR_UNSUPPORTED", 3: "BLK_ERR_ALIGNMENT",
                4: "BLK_ERR_CACHE_FULL", 5: "BLK_ERR_CUDA", 6: "BLK_ERR_TIMEOUT", 7: "BLK_ERR_WORKSPACE"}
ACTS = {"silu": 0, "swiglu": 0, "relu2": 1, "xielu": 2}
DTYPES = {"f32": 0, "fp32": 0, "float32": 0, "bf16": 1, "bfloat16": 1}


class blk_desc(ctypes.Structure):
    _fields_ = [("hidden", c_int), ("n_heads", c_int), ("n_kv_heads", c_int), ("head_dim", c_int), ("ffn", c_int),
                ("rope_theta", c_float), ("eps", c_float), ("act", c_int), ("xielu_alpha_p", c_float),
                ("xielu_alpha_n", c_float), ("xielu_beta", c_float), ("xielu_eps", c_float), ("qk_norm", c_int),
                ("dtype", c_int), ("max_batch", c_int), ("max_seq", c_int), ("rope_type", c_int),
                ("rope_factor", c_float), ("rope_orig_max_pos", c_int), ("rope_low", c_float), ("rope_high", c_float),
                ("sliding_window", c_int), ("no_rope", c_int), ("attn_gate", c_int), ("sandwich_norm", c_int)]

ROPE_TYPES = {"yarn": 1, "llama3": 2}


class blk_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("ln1_g", "wq", "wk", "wv", "q_norm_g", "k_norm_g", "wo", "ln2_g",
                                         "w_gate", "w_up", "w_down", "prepared", "w_attn_gate", "post_attn_g",
                                         "post_mlp_g")]


class blk_kv_cache(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("capacity", c_int), ("lens", c_void_p)]


class blk_model(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("layers", POINTER(blk_weights)), ("n_layers", c_int), ("norm_g", c_void_p),
                ("lm_head", c_void_p), ("vocab", c_int)]


TAP_NAMES = ("attention_queries", "attention_keys", "attention_values", "attention_head_outputs",
             "attention_output", "layer_mid", "mlp_neurons", "mlp_output")


class blk_taps(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in TAP_NAMES]


# name -> (restype, argtypes); the exported symbols of include/blk.h
SIGNATURES = {
    "blk_create": (c_int, [POINTER(blk_desc), POINTER(c_void_p)]),
    "blk_destroy": (c_int, [c_void_p]),
    "blk_workspace_bytes": (c_size_t, [c_void_p, c_int, c_int, c_int]),
    "blk_forward": (c_int, [c_void_p, c_void_p, c_int, c_int, POINTER(blk_weights), POINTER(blk_kv_cache), c_int,
                            c_void_p, c_void_p, c_size_t, POINTER(blk_taps), c_void_p]),
    "blk_forward_masked": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, POINTER(blk_weights), c_void_p,
                                   c_void_p, c_size_t, POINTER(blk_taps), c_void_p]),
    "blk_rmsnorm": (c_int, [c_void_p, c_void_p, c_int, c_int, c_float, c_void_p, c_int, c_void_p]),
    "blk_qkv_rope": (c_int, [c_void_p, c_void_p, POINTER(blk_weights), c_int, c_int, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_size_t, c_void_p]),
    "blk_attn_gqa": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                             c_void_p, c_size_t, c_void_p]),
    "blk_mlp": (c_int, [c_void_p, c_void_p, c_void_p, POINTER(blk_weights), c_int, c_void_p, c_void_p, c_size_t,
                        c_void_p]),
    "blk_stage_workspace_bytes": (c_size_t, [c_void_p, c_int]),
    "blk_last_status": (c_int, [c_void_p]),
    "blk_xielu_effective": (None, [c_float, c_float, c_float, POINTER(c_float), POINTER(c_float)]),
    "blk_error_string": (c_char_p, [c_int]),
    "blk_last_error_message": (c_char_p, []),
    "blk_debug_set_wait_timeout_ns": (None, [c_longlong]),
    "blk_debug_last_status": (c_int, []),
    "blk_version": (c_char_p, []),
    "blk_profile_enable": (c_int, [c_void_p, c_int]),
    "blk_profile_collect": (c_int, [c_void_p, POINTER(ctypes.c_double), POINTER(c_longlong), c_int]),
    "blk_profile_stage_name": (c_char_p, [c_void_p, c_int]),
    "blk_profile_reset": (None, [c_void_p]),
    "blk_debug_gemm_bf16": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                    c_void_p]),
    "blk_forward_graph_create": (c_int, [c_void_p, c_void_p, c_int, c_int, POINTER(blk_weights),
                                         POINTER(blk_kv_cache), c_int, c_void_p, c_void_p, c_size_t,
                                         POINTER(blk_taps), POINTER(c_void_p)]),
    "blk_graph_launch": (c_int, [c_void_p, c_void_p]),
    "blk_graph_destroy": (c_int, [c_void_p]),
    "blk_prepared_bytes": (c_size_t, [c_void_p]),
    "blk_prepare_weights": (c_int, [c_void_p, POINTER(blk_weights), c_void_p, c_size_t, c_void_p]),
    "blk_attn_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                        c_void_p, c_void_p]),
    "blk_model_workspace_bytes": (c_size_t, [c_void_p, c_int, c_int, c_int]),
    "blk_model_forward": (c_int, [c_void_p, POINTER(blk_model), c_void_p, c_int, c_int, POINTER(blk_kv_cache), c_int,
                                  c_void_p, c_void_p, c_size_t, c_void_p]),
}

_lib_handle = None


def lib():
    """Loads libblk.so (once). Raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(python -m llama_family_decoder_gb300.build)")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = h
    return _lib_handle


class BlkError(RuntimeError):
    def __init__(self, status, msg=""):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")


def _check(status):
    if status != BLK_OK:
        raise BlkError(status, lib().blk_last_error_message().decode())


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


def xielu_effective(raw_alpha_p, raw_alpha_n, beta=0.5):
    ap, an = c_float(), c_float()
    lib().blk_xielu_effective(raw_alpha_p, raw_alpha_n, beta, ctypes.byref(ap), ctypes.byref(an))
    return ap.value, an.value


def set_wait_timeout_ns(ns: int):
    lib().blk_debug_set_wait_timeout_ns(int(ns))


def make_weights_struct(w: dict) -> blk_weights:
    """Page-named weight tensors (input_layernorm, q_proj, ...) -> blk_weights.

    The "afmoe" weights: attn_gate_proj (the attention gate), post_attn_norm and
    post_mlp_norm (the sandwich post-norms); post_attention_layernorm stays the
    MLP's input norm."""
    g = w.get
    return blk_weights(_ptr(g("input_layernorm")), _ptr(g("q_proj")), _ptr(g("k_proj")), _ptr(g("v_proj")),
                       _ptr(g("q_norm")), _ptr(g("k_norm")), _ptr(g("o_proj")), _ptr(g("post_attention_layernorm")),
                       _ptr(g("gate_proj")), _ptr(g("up_proj")), _ptr(g("down_proj")), _ptr(g("prepared")),
                       _ptr(g("attn_gate_proj")), _ptr(g("post_attn_norm")), _ptr(g("post_mlp_norm")))


class DecoderBlock:
    """One decoder block handle (blk_create) and its calls."""

    def __init__(self, hidden, n_heads, n_kv_heads, head_dim, ffn, act="silu", dtype="bf16", qk_norm=False,
                 rope_theta=10000.0, eps=1e-5, xielu_alpha_p=0.8, xielu_alpha_n=0.8, xielu_beta=0.5,
                 xielu_eps=-1e-6, max_batch=64, max_seq=4096, rope_scaling=None, sliding_window=0, use_rope=True,
                 attn_gate=False, sandwich_norm=False):
        # rope_scaling: None, or (kind, factor, original_max_position, low, high), kind "yarn" | "llama3"
        rs = (ROPE_TYPES[rope_scaling[0]], *rope_scaling[1:]) if rope_scaling else (0, 1.0, 0, 0.0, 0.0)
        self.desc = blk_desc(hidden, n_heads, n_kv_heads, head_dim, ffn, rope_theta, eps, ACTS[act],
                             xielu_alpha_p, xielu_alpha_n, xielu_beta, xielu_eps, int(bool(qk_norm)), DTYPES[dtype],
                             max_batch, max_seq, rs[0], float(rs[1]), int(rs[2]), float(rs[3]), float(rs[4]),
                             int(sliding_window), int(not use_rope), int(bool(attn_gate)), int(bool(sandwich_norm)))
        h = c_void_p()
        _check(lib().blk_create(ctypes.byref(self.desc), ctypes.byref(h)))
        self.handle = h
        self._ws = None

    @classmethod
    def from_workload(cls, wl, max_batch=None, max_seq=None):
        return cls(wl.hidden_size, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.intermediate_size,
                   act=wl.hidden_act, dtype=wl.dtype, qk_norm=wl.qk_norm, rope_theta=wl.rope_theta,
                   eps=wl.rms_norm_eps, xielu_alpha_p=wl.xielu_alpha_p, xielu_alpha_n=wl.xielu_alpha_n,
                   max_batch=max_batch or wl.batch, max_seq=max_seq or wl.cache_len + wl.seq,
                   rope_scaling=wl.rope_scaling, sliding_window=wl.sliding_window, use_rope=wl.use_rope,
                   attn_gate=wl.attn_gate, sandwich_norm=wl.sandwich_norm)

    def close(self):
        if self.handle:
            lib().blk_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prepare(self, weights, stream=None):
        """fp16 copies of wo / w_gate / w_up (blk_prepare_weights); returns weights plus 'prepared'."""
        import torch
        buf = torch.empty(max(lib().blk_prepared_bytes(self.handle), 16), dtype=torch.uint8,
                          device=weights["o_proj"].device)
        wst = make_weights_struct(weights)
        _check(lib().blk_prepare_weights(self.handle, ctypes.byref(wst), _ptr(buf), buf.numel(), _stream_ptr(stream)))
        return dict(weights, prepared=buf)

    def model_workspace_bytes(self, batch, seq, decode=False):
        return lib().blk_model_workspace_bytes(self.handle, batch, seq, int(bool(decode)))

    def workspace_bytes(self, batch, seq, decode=False):
        return lib().blk_workspace_bytes(self.handle, batch, seq, int(decode))

    def stage_workspace_bytes(self, rows):
        return lib().blk_stage_workspace_bytes(self.handle, rows)

    def _workspace(self, nbytes, device):
        import torch
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        return self._ws

    def forward(self, x, weights, cache=None, out=None, workspace=None, taps=None, stream=None, host_lens_max=-1,
                attention_mask=None):
        """out = block(x); x [B, T, D] device tensor. cache: dict(k, v, lens): T new tokens per
        sequence after lens[b] cached positions (a decode step for T == 1, a prefill chunk for
        T > 1, which needs host_lens_max = max(lens)). attention_mask: device int32 [B, T] of a
        padded prefill batch (blk_forward_masked; zeros are padding)."""
        import torch
        B, T, _ = x.shape
        if out is None:
            out = torch.empty_like(x)
        need = self.workspace_bytes(B, T, cache is not None)
        if workspace is None:
            workspace = self._workspace(need, x.device)
        ws_bytes = workspace.numel() * workspace.element_size()
        wst = weights if isinstance(weights, blk_weights) else make_weights_struct(weights)
        kvc = None
        if cache is not None:
            kvc = blk_kv_cache(_ptr(cache["k"]), _ptr(cache["v"]), cache["k"].shape[2], _ptr(cache["lens"]))
        tp = None
        if taps:
            tp = blk_taps(*[_ptr(taps.get(n)) for n in TAP_NAMES])
        if attention_mask is not None:
            if cache is not None:
                raise ValueError("attention_mask: prefill batches only")
            _check(lib().blk_forward_masked(self.handle, _ptr(x), B, T, _ptr(attention_mask), ctypes.byref(wst),
                                            _ptr(out), _ptr(workspace), ws_bytes,
                                            ctypes.byref(tp) if tp is not None else None, _stream_ptr(stream)))
            return out
        _check(lib().blk_forward(self.handle, _ptr(x), B, T, ctypes.byref(wst),
                                 ctypes.byref(kvc) if kvc is not None else None, int(host_lens_max), _ptr(out),
                                 _ptr(workspace), ws_bytes, ctypes.byref(tp) if tp is not None else None,
                                 _stream_ptr(stream)))
        return out

    def model_forward(self, tokens, layers, embed, norm_g, lm_head, caches=None, host_lens_max=-1, logits=None,
                      workspace=None, stream=None):
        """logits [B, T, vocab] of the model around this block's shape: embed[tokens], the
        layers (a list of weight dicts), the final norm and lm_head. tokens: device int32
        [B, T]. caches: None, or one dict(k, v, lens) per layer (T new tokens after lens)."""
        import torch
        B, T = tokens.shape
        vocab = embed.shape[0]
        if logits is None:
            logits = torch.empty(B, T, vocab, dtype=embed.dtype, device=tokens.device)
        need = lib().blk_model_workspace_bytes(self.handle, B, T, int(caches is not None))
        if workspace is None:
            workspace = self._workspace(need, tokens.device)
        wls = (blk_weights * len(layers))(*[make_weights_struct(w) for w in layers])
        m = blk_model(_ptr(embed), wls, len(layers), _ptr(norm_g), _ptr(lm_head), vocab)
        kvs = None
        if caches is not None:
            kvs = (blk_kv_cache * len(caches))(*[blk_kv_cache(_ptr(c["k"]), _ptr(c["v"]), c["k"].shape[2],
                                                              _ptr(c["lens"])) for c in caches])
        _check(lib().blk_model_forward(self.handle, ctypes.byref(m), _ptr(tokens), B, T, kvs, host_lens_max,
                                       _ptr(logits), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream_ptr(stream)))
        return logits

    def forward_graph(self, x, weights, out, workspace, cache=None, taps=None, host_lens_max=-1):
        """Records blk_forward for these exact buffers into a CUDA graph (ForwardGraph)."""
        B, T, _ = x.shape
        wst = weights if isinstance(weights, blk_weights) else make_weights_struct(weights)
        kvc = None
        if cache is not None:
            kvc = blk_kv_cache(_ptr(cache["k"]), _ptr(cache["v"]), cache["k"].shape[2], _ptr(cache["lens"]))
        tp = blk_taps(*[_ptr(taps.get(n)) for n in TAP_NAMES]) if taps else None
        g = c_void_p()
        _check(lib().blk_forward_graph_create(self.handle, _ptr(x), B, T, ctypes.byref(wst),
                                              ctypes.byref(kvc) if kvc is not None else None, int(host_lens_max),
                                              _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                              ctypes.byref(tp) if tp is not None else None, ctypes.byref(g)))
        return ForwardGraph(g, keep=(x, weights, out, workspace, cache, taps, wst, kvc, tp))

    def qkv_rope(self, y, weights, batch, seq, q, k, v, pos0=None, stream=None):
        need = self.stage_workspace_bytes(batch * seq)
        ws = self._workspace(need, y.device)
        wst = make_weights_struct(weights)
        _check(lib().blk_qkv_rope(self.handle, _ptr(y), ctypes.byref(wst), batch, seq, _ptr(pos0), _ptr(q), _ptr(k),
                                  _ptr(v), _ptr(ws), ws.numel(), _stream_ptr(stream)))

    def attn_gqa(self, q, k, v, o, kv_lens=None, stream=None):
        B, H, Tq, _ = q.shape
        kv_stride = k.shape[2]
        ws = self._workspace(self.stage_workspace_bytes(B * Tq), q.device)
        _check(lib().blk_attn_gqa(self.handle, _ptr(q), _ptr(k), _ptr(v), B, Tq, kv_stride, _ptr(kv_lens), _ptr(o),
                                  _ptr(ws), ws.numel(), _stream_ptr(stream)))

    def mlp(self, resid, h_normed, weights, out, stream=None):
        rows = resid.numel() // resid.shape[-1]
        ws = self._workspace(self.stage_workspace_bytes(rows), resid.device)
        wst = make_weights_struct(weights)
        _check(lib().blk_mlp(self.handle, _ptr(resid), _ptr(h_normed), ctypes.byref(wst), rows, _ptr(out), _ptr(ws),
                             ws.numel(), _stream_ptr(stream)))

    def last_status(self):
        return lib().blk_last_status(self.handle)

    def profile(self, on=True):
        _check(lib().blk_profile_enable(self.handle, int(bool(on))))

    def profile_reset(self):
        lib().blk_profile_reset(self.handle)

    def profile_collect(self):
        """Waits for the last profiled forward; returns {stage: (total_ms, launches)}."""
        n_max = 24
        ms = (ctypes.c_double * n_max)()
        ln = (c_longlong * n_max)()
        n = lib().blk_profile_collect(self.handle, ms, ln, n_max)
        if n < 0:
            raise BlkError(5, "profiling is off or a CUDA error occurred")
        return {lib().blk_profile_stage_name(self.handle, i).decode(): (ms[i], ln[i]) for i in range(n)}


class ForwardGraph:
    """A recorded blk_forward (blk_graph); launch() replays it on a stream."""

    def __init__(self, handle, keep):
        self.handle = handle
        self._keep = keep  # the buffers the graph reads and writes stay alive with it

    def launch(self, stream=None):
        _check(lib().blk_graph_launch(self.handle, _stream_ptr(stream)))

    def close(self):
        if self.handle:
            lib().blk_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def rmsnorm(x, g, eps=1e-5, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty_like(x)
    n = x.shape[-1]
    rows = x.numel() // n
    dt = 1 if x.dtype == torch.bfloat16 else 0
    _check(lib().blk_rmsnorm(_ptr(x), _ptr(g), rows, n, eps, _ptr(out), dt, _stream_ptr(stream)))
    return out


def debug_gemm_bf16(a, b, bn=256, split_k=1, out=None, stream=None, pair=False):
    """c = a @ b.T on the bare tcgen05 GEMM (bf16 out), or fp32 split-K partials [split, N, M];
    pair: CTA pairs with 256-row tiles."""
    import torch
    M, K = a.shape
    N = b.shape[0]
    if out is None:
        if split_k == 1:
            out = torch.empty(M, N, dtype=torch.bfloat16, device=a.device)
        else:
            out = torch.empty(split_k, M, N, dtype=torch.float32, device=a.device)
    _check(lib().blk_debug_gemm_bf16(_ptr(a), _ptr(b), _ptr(out), M, N, K, bn, split_k, 1 if pair else 0,
                                     _stream_ptr(stream)))
    return out


def attn_decode_noalloc(q, k, v, kv_lens, o, stream=None):
    """Decode attention through blk_attn_decode_noalloc (no workspace, no handle).

    q [B, H, 1, d], k/v [B, Hkv, kv_stride, d], kv_lens int32 [B], o [B, 1, H, d]; bf16 on the device.
    """
    B, H = q.shape[0], q.shape[1]
    Hkv, kv_stride, d = k.shape[1], k.shape[2], k.shape[3]
    _check(lib().blk_attn_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_lens), B, H, Hkv, d, kv_stride, _ptr(o),
                                         _stream_ptr(stream)))
    return o
