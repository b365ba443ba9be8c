"""Thin Python binding of libekv.so (ctypes).  Argument marshalling only: every
step of the decode path runs in the library's CUDA kernels.  PyTorch supplies
device memory (through the caching allocator) and streams.

The binding never falls back to anything else: if libekv.so has not been
built, `lib()` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

BITS = (2, 4, 8, 16)
_CODE = {2: 0, 4: 1, 8: 2, 16: 3}
NUM_FORMATS = 16
AFTER_OTHER_LAYER = 1  # ekv_append_decode_attn flags
AFTER_PRODUCER = 2
DEBUG_WAIT_EXPIRY = 1  # ekv_debug_set knob


def fmt_index(k_bits: int, v_bits: int) -> int:
    return _CODE[k_bits] * 4 + _CODE[v_bits]


class EkvConfig(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32),
        ("max_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("pool_pages", ctypes.c_int64 * NUM_FORMATS),
        ("softmax_scale", ctypes.c_float),
        ("ema_alpha", ctypes.c_float),
        ("tau", ctypes.c_float),
        ("tau_ctx0", ctypes.c_int32),
        ("hysteresis", ctypes.c_float),
        ("vote", ctypes.c_int32),
        ("quantizer", ctypes.c_int32),
        ("dev_alloc", ctypes.c_void_p),
        ("dev_free", ctypes.c_void_p),
        ("alloc_ctx", ctypes.c_void_p),
    ]


class EkvStats(ctypes.Structure):
    _fields_ = [
        ("sealed_pages", ctypes.c_int64 * NUM_FORMATS),
        ("open_pages", ctypes.c_int64 * NUM_FORMATS),
        ("open_rows", ctypes.c_int64 * NUM_FORMATS),
        ("tokens", ctypes.c_int64),
        ("k_bits", ctypes.c_double),
        ("v_bits", ctypes.c_double),
        ("cost_vs_c0", ctypes.c_double),
        ("page_bytes", ctypes.c_double),
        ("fp16_bytes", ctypes.c_double),
        ("saved_vs_fp16", ctypes.c_double),
    ]


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p)

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SIGS = {
    "ekv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ekv_page_bytes": (_I32, [_I32, _I32, _I32]),
    "ekv_page_bytes_q": (_I32, [_I32, _I32, _I32, _I32]),
    "ekv_create": (ctypes.c_int, [ctypes.POINTER(EkvConfig), _P, _P, ctypes.POINTER(_P)]),
    "ekv_destroy": (ctypes.c_int, [_P]),
    "ekv_seq_reset": (ctypes.c_int, [_P, _I32, _P]),
    "ekv_append": (ctypes.c_int, [_P, _I32, _I32, _P, _I32, _P, _P, _P]),
    "ekv_decode_attn": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _P]),
    "ekv_append_decode_attn": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _P, _P, _I32, _P]),
    "ekv_decode_attn_noalloc": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _P]),
    "ekv_canary_kl": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _P]),
    "ekv_canary_kl_layers": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, ctypes.c_int64, _P,
                                            _P]),
    "ekv_tier_update": (ctypes.c_int, [_P, _P, _P, _I32, _P]),
    "ekv_set_tiers": (ctypes.c_int, [_P, _P, _P]),
    "ekv_get_state": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "ekv_seq_len": (ctypes.c_int, [_P, _I32, _I32, _P, _P]),
    "ekv_block_table": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _I32, _P, _P]),
    "ekv_read_pages": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _I32, _P, ctypes.c_size_t, _P]),
    "ekv_pool_free": (ctypes.c_int, [_P, _I32, _P, _P]),
    "ekv_stats": (ctypes.c_int, [_P, _I32, _I32, ctypes.POINTER(EkvStats), _P]),
    "ekv_debug_set": (ctypes.c_int, [_P, _I32, ctypes.c_int64]),
    "ekv_sync": (ctypes.c_int, [_P, _P]),
    "ekv_state_size": (ctypes.c_int64, [_P]),
    "ekv_state_save": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P]),
    "ekv_state_load": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P]),
    "ekv_set_clip": (ctypes.c_int, [_P, _I32, _P, _P, _P]),
    "ekv_get_clip": (ctypes.c_int, [_P, _I32, _P, _P, _P]),
    "ekv_abs_percentile": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int64, _I32,
                                          ctypes.c_int64, _I32, ctypes.c_double, _P, _P,
                                          ctypes.c_int64, _P]),
    "ekv_abs_percentile_scratch_bytes": (ctypes.c_int, [_I32, _P]),
    "ekv_autok": (ctypes.c_int, [_P, _I32, ctypes.c_double, _P, _P]),
    "ekv_output_error": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P, _P, _P]),
}
EXPORTS = tuple(_SIGS)

_LIB = None


def lib() -> ctypes.CDLL:
    """Load libekv.so; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


class EkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {lib().ekv_status_string(code).decode()} (status {code})")


def _check(rc: int, what: str):
    if rc != 0:
        raise EkvError(rc, what)


QUANT_SYMMETRIC, QUANT_ASYMMETRIC = 0, 1


def page_bytes(k_bits: int, v_bits: int, head_dim: int, asym: bool = False) -> int:
    return lib().ekv_page_bytes_q(k_bits, v_bits, head_dim,
                                  QUANT_ASYMMETRIC if asym else QUANT_SYMMETRIC)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Cache:
    """One handle of the library: paged mixed-precision KV cache of all layers."""

    def __init__(self, num_layers: int, max_seqs: int, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, max_seq_len: int, pool_pages: dict, k_bits_init, v_bits,
                 alpha: float = 0.25, tau: float = 0.05, softmax_scale: float = 0.0,
                 device=None, torch_alloc: bool = True, tau_ctx0: int = 0,
                 hysteresis: float = 0.0, vote: int = 1, asym: bool = False):
        L = lib()
        self.device = torch.device("cuda" if device is None else device)
        self.num_layers, self.max_seqs = num_layers, max_seqs
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, num_kv_heads, head_dim
        self.v_bits = [int(b) for b in v_bits]
        cfg = EkvConfig()
        cfg.num_layers, cfg.max_seqs = num_layers, max_seqs
        cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim = num_q_heads, num_kv_heads, head_dim
        cfg.max_seq_len = max_seq_len
        for (kb, vb), n in pool_pages.items():
            cfg.pool_pages[fmt_index(kb, vb)] = int(n)
        cfg.softmax_scale, cfg.ema_alpha, cfg.tau = softmax_scale, alpha, tau
        cfg.tau_ctx0, cfg.hysteresis, cfg.vote = int(tau_ctx0), float(hysteresis), int(vote)
        cfg.quantizer = QUANT_ASYMMETRIC if asym else QUANT_SYMMETRIC
        self.asym = bool(asym)
        self._keep = []
        if torch_alloc:
            dev = self.device.index if self.device.index is not None else torch.cuda.current_device()

            def _alloc(nbytes, ctx):
                return torch.cuda.caching_allocator_alloc(int(nbytes), dev)

            def _free(p, ctx):
                torch.cuda.caching_allocator_delete(p)

            a, f = ALLOC_FN(_alloc), FREE_FN(_free)
            self._keep += [a, f]
            cfg.dev_alloc = ctypes.cast(a, ctypes.c_void_p)
            cfg.dev_free = ctypes.cast(f, ctypes.c_void_p)
        kb = (ctypes.c_uint8 * num_layers)(*[int(b) for b in k_bits_init])
        vb = (ctypes.c_uint8 * num_layers)(*self.v_bits)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(L.ekv_create(ctypes.byref(cfg), kb, vb, ctypes.byref(h)), "ekv_create")
        self._h = h

    # ---- lifecycle ------------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None):
            lib().ekv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    # ---- hot path ---------------------------------------------------------------
    def append(self, layer: int, seq_slots: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
               stream=None):
        n_seqs = seq_slots.numel()
        n_new = k.shape[1] if n_seqs else 1
        _check(lib().ekv_append(self._h, layer, n_seqs, _ptr(seq_slots), n_new, _ptr(k), _ptr(v),
                                _stream(stream)), "ekv_append")

    def decode_attn(self, layer: int, seq_slots: torch.Tensor, q: torch.Tensor,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(q)
        _check(lib().ekv_decode_attn(self._h, layer, seq_slots.numel(), _ptr(seq_slots), _ptr(q),
                                     _ptr(out), _stream(stream)), "ekv_decode_attn")
        return out

    def append_decode_attn(self, layer: int, seq_slots: torch.Tensor, k: torch.Tensor,
                           v: torch.Tensor, q: torch.Tensor, out: torch.Tensor | None = None,
                           after_other_layer: bool = False, after_producer: bool = False,
                           stream=None) -> torch.Tensor:
        """One decode step of a layer in one launch: append one token (k, v of shape
        [n, 1, Hkv, d] or [n, Hkv, d]) to every sequence, then attend over it too.
        `after_other_layer`: the previous work on the stream is this call for
        another layer and writes none of this call's inputs; `after_producer`:
        the previous work may write q, k, v (but not this layer's cache).  Either
        lets the launch overlap its start with that work's end."""
        if out is None:
            out = torch.empty_like(q)
        flags = ((AFTER_OTHER_LAYER if after_other_layer else 0) |
                 (AFTER_PRODUCER if after_producer else 0))
        _check(lib().ekv_append_decode_attn(self._h, layer, seq_slots.numel(), _ptr(seq_slots),
                                            _ptr(k), _ptr(v), _ptr(q), _ptr(out), flags,
                                            _stream(stream)), "ekv_append_decode_attn")
        return out

    def decode_attn_noalloc(self, layer: int, seq_slots: torch.Tensor, q: torch.Tensor,
                            out: torch.Tensor, stream=None) -> torch.Tensor:
        """Decode attention with the library's static scratch (no allocation at all)."""
        _check(lib().ekv_decode_attn_noalloc(self._h, layer, seq_slots.numel(), _ptr(seq_slots),
                                             _ptr(q), _ptr(out), _stream(stream)),
               "ekv_decode_attn_noalloc")
        return out

    def canary_kl(self, layer: int, seq_slots: torch.Tensor, q: torch.Tensor,
                  delta_out: torch.Tensor | None = None, stream=None):
        _check(lib().ekv_canary_kl(self._h, layer, seq_slots.numel(), _ptr(seq_slots), _ptr(q),
                                   _ptr(delta_out), _stream(stream)), "ekv_canary_kl")
        return delta_out

    def canary_kl_layers(self, first_layer: int, seq_slots: torch.Tensor, q: torch.Tensor,
                         delta_out: torch.Tensor | None = None, stream=None):
        """Canary of layers first_layer .. first_layer + q.shape[0] - 1 in one launch;
        q [n_layers, n_seqs, Hq, d] (each layer's block contiguous)."""
        n = q.shape[0]
        if q[0].numel() and not q[0].is_contiguous():
            raise ValueError("each layer's queries must be contiguous")
        stride = q.stride(0) if n > 1 else 0
        _check(lib().ekv_canary_kl_layers(self._h, first_layer, n, seq_slots.numel(),
                                          _ptr(seq_slots), _ptr(q), stride, _ptr(delta_out),
                                          _stream(stream)), "ekv_canary_kl_layers")
        return delta_out

    def tier_update(self, delta: torch.Tensor | None = None, layer_mask: torch.Tensor | None = None,
                    freeze: bool = False, stream=None):
        _check(lib().ekv_tier_update(self._h, _ptr(delta), _ptr(layer_mask), int(freeze),
                                     _stream(stream)), "ekv_tier_update")

    # ---- control and inspection ------------------------------------------------
    def set_clip(self, layer: int, k_clip=None, v_clip=None, stream=None):
        """Load one layer's clipping thresholds: k_clip [Hkv, d], v_clip [Hkv]
        (anything float-convertible; None = no clipping for that part)."""
        H, d = self.num_kv_heads, self.head_dim

        def arr(x, n):
            if x is None:
                return None
            v = [float(t) for t in torch.as_tensor(x, dtype=torch.float32).reshape(-1).tolist()]
            if len(v) != n:
                raise ValueError(f"expected {n} thresholds, got {len(v)}")
            return (ctypes.c_float * n)(*v)

        _check(lib().ekv_set_clip(self._h, layer, arr(k_clip, H * d), arr(v_clip, H),
                                  _stream(stream)), "ekv_set_clip")

    def get_clip(self, layer: int, stream=None):
        """(k_clip [Hkv, d], v_clip [Hkv]) float32 CPU tensors (+inf: none)."""
        H, d = self.num_kv_heads, self.head_dim
        k = (ctypes.c_float * (H * d))()
        v = (ctypes.c_float * H)()
        _check(lib().ekv_get_clip(self._h, layer, k, v, _stream(stream)), "ekv_get_clip")
        return (torch.tensor(list(k), dtype=torch.float32).view(H, d),
                torch.tensor(list(v), dtype=torch.float32))

    def set_tiers(self, tiers, stream=None):
        t = (ctypes.c_uint8 * self.num_layers)(*[int(b) for b in tiers])
        _check(lib().ekv_set_tiers(self._h, t, _stream(stream)), "ekv_set_tiers")

    def state(self, stream=None) -> dict:
        L = self.num_layers
        t = (ctypes.c_uint8 * L)()
        e = (ctypes.c_float * (3 * L))()
        d = (ctypes.c_float * (3 * L))()
        v = (ctypes.c_int32 * L)()
        _check(lib().ekv_get_state(self._h, t, e, d, v, _stream(stream)), "ekv_get_state")
        return {"tiers": list(t), "ema": [list(e[3 * i:3 * i + 3]) for i in range(L)],
                "delta": [list(d[3 * i:3 * i + 3]) for i in range(L)], "ema_valid": list(v)}

    def stats(self, first_layer: int = 0, n_layers: int | None = None, stream=None) -> dict:
        """What the cache of the given layers holds (ekv_stats): pages per format,
        mean stored K/V bits per element, page bytes against fp16."""
        n = self.num_layers - first_layer if n_layers is None else n_layers
        out = EkvStats()
        _check(lib().ekv_stats(self._h, first_layer, n, ctypes.byref(out), _stream(stream)),
               "ekv_stats")
        d = {name: getattr(out, name) for name, _ in EkvStats._fields_}
        for k in ("sealed_pages", "open_pages", "open_rows"):
            d[k] = list(d[k])
        return d

    def seq_len(self, layer: int, slot: int, stream=None) -> int:
        out = ctypes.c_int32()
        _check(lib().ekv_seq_len(self._h, layer, slot, ctypes.byref(out), _stream(stream)),
               "ekv_seq_len")
        return out.value

    def block_table(self, layer: int, slot: int, kv_head: int, stream=None) -> list:
        n = ctypes.c_int32()
        _check(lib().ekv_block_table(self._h, layer, slot, kv_head, None, 0, ctypes.byref(n),
                                     _stream(stream)), "ekv_block_table")
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check(lib().ekv_block_table(self._h, layer, slot, kv_head, buf, n.value, ctypes.byref(n),
                                     _stream(stream)), "ekv_block_table")
        return list(buf[:n.value])

    def read_pages(self, layer: int, slot: int, kv_head: int, first: int, n: int,
                   stream=None) -> torch.Tensor:
        stride = page_bytes(16, 16, self.head_dim, self.asym)
        dst = torch.zeros(max(1, n), stride, dtype=torch.uint8, device=self.device)
        _check(lib().ekv_read_pages(self._h, layer, slot, kv_head, first, n, _ptr(dst), stride,
                                    _stream(stream)), "ekv_read_pages")
        return dst[:n]

    def pool_free(self, k_bits: int, v_bits: int, stream=None) -> int:
        out = ctypes.c_int64()
        _check(lib().ekv_pool_free(self._h, fmt_index(k_bits, v_bits), ctypes.byref(out),
                                   _stream(stream)), "ekv_pool_free")
        return out.value

    def reset(self, slot: int, stream=None):
        _check(lib().ekv_seq_reset(self._h, slot, _stream(stream)), "ekv_seq_reset")

    def debug_set(self, knob: int, value: int):
        """Set a test hook (ekv_debug_set; DEBUG_WAIT_EXPIRY)."""
        _check(lib().ekv_debug_set(self._h, knob, int(value)), "ekv_debug_set")

    def sync(self, stream=None):
        """Wait for the stream and raise if a kernel recorded a device-side error."""
        _check(lib().ekv_sync(self._h, _stream(stream)), "device error")

    def save_state(self, stream=None) -> bytes:
        n = lib().ekv_state_size(self._h)
        buf = ctypes.create_string_buffer(n)
        _check(lib().ekv_state_save(self._h, buf, n, _stream(stream)), "ekv_state_save")
        return buf.raw

    def load_state(self, blob: bytes, stream=None):
        _check(lib().ekv_state_load(self._h, blob, len(blob), _stream(stream)), "ekv_state_load")


def abs_percentile(x: torch.Tensor, q: float, n_rows: int, row_stride: int, n_groups: int,
                   group_stride: int, group_width: int, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """Nearest-rank q-quantile of |x| per group (ekv_abs_percentile) -> float32 [n_groups]."""
    if x.dtype != torch.float16 or not x.is_cuda:
        raise TypeError("x must be a CUDA fp16 tensor")
    if out is None:
        out = torch.empty(n_groups, dtype=torch.float32, device=x.device)
    nb = ctypes.c_int64(0)
    if n_groups >= 1:
        _check(lib().ekv_abs_percentile_scratch_bytes(n_groups, ctypes.byref(nb)),
               "ekv_abs_percentile_scratch_bytes")
    scratch = torch.empty(max(4, nb.value) // 4, dtype=torch.int32, device=x.device)
    _check(lib().ekv_abs_percentile(_ptr(x), n_rows, row_stride, n_groups, group_stride,
                                    group_width, float(q), _ptr(out), _ptr(scratch), nb.value,
                                    _stream(stream)), "ekv_abs_percentile")
    return out


def k_thresholds(k: torch.Tensor, q: float, stream=None) -> torch.Tensor:
    """Per (KV head, channel) thresholds [Hkv, d] of contiguous keys [T, Hkv, d]."""
    T, H, d = k.shape
    k = k.contiguous()
    return abs_percentile(k, q, T, H * d, H * d, 1, 1, stream=stream).view(H, d)


def v_thresholds(v: torch.Tensor, q: float, stream=None) -> torch.Tensor:
    """Per KV head thresholds [Hkv] of contiguous values [T, Hkv, d]."""
    T, H, d = v.shape
    v = v.contiguous()
    return abs_percentile(v, q, T, H * d, H, d, d, stream=stream)


def output_error(o_hat: torch.Tensor, o_ref: torch.Tensor, stream=None):
    """(sum (o_hat - o_ref)^2, sum o_ref^2) over two fp16 CUDA tensors of one
    shape, in fp64 on the GPU (ekv_output_error)."""
    if o_hat.shape != o_ref.shape or o_hat.dtype != torch.float16 or o_ref.dtype != torch.float16:
        raise TypeError("two fp16 tensors of one shape")
    a, b = o_hat.contiguous(), o_ref.contiguous()
    scratch = torch.empty(2, dtype=torch.float64, device=a.device)
    out = (ctypes.c_double * 2)()
    _check(lib().ekv_output_error(_ptr(a), _ptr(b), a.numel(), out, _ptr(scratch),
                                  _stream(stream)), "ekv_output_error")
    return out[0], out[1]


def autok(sensitivity, frac: float):
    """(k, order): the fewest most-sensitive layers holding >= frac of the total."""
    s = [float(x) for x in sensitivity]
    n = len(s)
    arr = (ctypes.c_double * max(1, n))(*s)
    order = (ctypes.c_int32 * max(1, n))()
    k = ctypes.c_int32()
    _check(lib().ekv_autok(arr, n, float(frac), order, ctypes.byref(k)), "ekv_autok")
    return k.value, list(order[:n])


def cache_for(w, device=None, max_seqs: int | None = None, torch_alloc: bool = True,
              **controller) -> Cache:
    """A cache sized for a `workloads.Workload`; `controller` passes the
    controller variants (tau_ctx0, hysteresis, vote)."""
    return Cache(w.num_layers, max_seqs or w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                 w.max_seq_len, w.pool_pages(), w.k_bits_init, w.v_bits, alpha=w.alpha,
                 tau=w.tau, device=device, torch_alloc=torch_alloc,
                 asym=getattr(w, "asym", False), **controller)
