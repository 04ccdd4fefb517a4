"""ctypes binding of libcsa.so: argument marshalling only.

Every function here checks each tensor's dtype and shape against the layer
and the call (the C ABI sees only untyped pointers, so a wrong dtype or shape
would otherwise be read as garbage) and that it is a contiguous CUDA tensor,
all before anything is allocated or enqueued; then it passes raw device
pointers and the current CUDA stream to the C ABI declared in include/csa.h
and turns a non-zero csa_status into an exception.  All arithmetic runs in the
library's CUDA kernels; there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libcsa.so")

CSA_F32, CSA_BF16 = 0, 1
OP_COMPRESS, OP_INDEX_TOPK, OP_ATTEND_DECODE, OP_ATTEND_PREFILL, OP_COMPRESS_PAIR = 0, 1, 2, 3, 4
OP_COMPRESS_VARLEN, OP_ATTEND_PREFILL_VARLEN = 5, 6
FP8_ROW_BYTES = 144  # CSA_FP8_ROW_BYTES: 128 E4M3 codes, the fp32 scale, 12 zero bytes
DEV_CAPACITY, DEV_STATE, DEV_RANGE, DEV_ROLLBACK = 1, 2, 4, 8
CSA_OK, CSA_ERR_ARG, CSA_ERR_UNSUPPORTED, CSA_ERR_CUDA, CSA_ERR_WORKSPACE = 0, 1, 2, 3, 4
STATUS = {0: "CSA_OK", 1: "CSA_ERR_ARG", 2: "CSA_ERR_UNSUPPORTED", 3: "CSA_ERR_CUDA", 4: "CSA_ERR_WORKSPACE"}
EXPORTS = ("csa_kernel_launches", "csa_frontier_slots", "csa_workspace_size", "csa_compress_append", "csa_index_topk",
           "csa_attend_decode", "csa_attend_prefill_chunk", "csa_status_string", "csa_static_scratch_bytes",
           "csa_index_topk_static", "csa_index_topk_overlapped", "csa_advance_positions",
           "csa_compress_append_pair", "csa_trim", "csa_index_topk_verify", "csa_attend_verify",
           "csa_compress_append_varlen", "csa_attend_prefill_varlen", "csa_index_rows_fp8")


class CSAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class _Layer(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("H", ctypes.c_int), ("D", ctypes.c_int), ("R", ctypes.c_int),
                ("W", ctypes.c_int), ("ratio", ctypes.c_int), ("Hi", ctypes.c_int), ("Di", ctypes.c_int),
                ("topk", ctypes.c_int), ("X", ctypes.c_int), ("scale", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("rollback", ctypes.c_int), ("index_fp8", ctypes.c_int)]


class _Comp(ctypes.Structure):
    _fields_ = [("wkv", ctypes.c_void_p), ("wgate", ctypes.c_void_p), ("ape", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p), ("d", ctypes.c_int)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libcsa.so (built by build.py); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"CSA CUDA library not built: {path} is missing "
                          "(run deepseek_v4_compressed_csa_gb300.build.build())")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.csa_frontier_slots.argtypes = [i32]
    lib.csa_frontier_slots.restype = i32
    lib.csa_kernel_launches.argtypes = []
    lib.csa_kernel_launches.restype = ctypes.c_ulonglong
    lib.csa_status_string.argtypes = [i32]
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_workspace_size.argtypes = [vp, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.csa_workspace_size.restype = i32
    lib.csa_compress_append.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, i32, vp, vp, vp, sz, vp, vp]
    lib.csa_compress_append.restype = i32
    lib.csa_index_topk.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.csa_index_topk.restype = i32
    lib.csa_index_topk_overlapped.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.csa_index_topk_overlapped.restype = i32
    lib.csa_static_scratch_bytes.argtypes = []
    lib.csa_static_scratch_bytes.restype = sz
    lib.csa_index_topk_static.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.csa_index_topk_static.restype = i32
    lib.csa_attend_decode.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.csa_attend_decode.restype = i32
    lib.csa_attend_prefill_chunk.argtypes = [vp, vp, vp, vp, vp, vp, i32, ctypes.c_int32, vp, vp, vp, i32, vp, vp,
                                             vp, vp, vp, sz, vp, vp]
    lib.csa_attend_prefill_chunk.restype = i32
    lib.csa_compress_append_pair.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, i32, vp, vp, vp, i32, vp, vp, vp,
                                             sz, vp, vp]
    lib.csa_compress_append_pair.restype = i32
    lib.csa_advance_positions.argtypes = [vp, i32, i32, vp]
    lib.csa_advance_positions.restype = i32
    lib.csa_trim.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.csa_trim.restype = i32
    lib.csa_index_topk_verify.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.csa_index_topk_verify.restype = i32
    lib.csa_attend_verify.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.csa_attend_verify.restype = i32
    lib.csa_compress_append_varlen.argtypes = [vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, i32, vp, vp, vp, sz, vp, vp]
    lib.csa_compress_append_varlen.restype = i32
    lib.csa_attend_prefill_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, vp, i32, vp, vp,
                                              vp, vp, vp, sz, vp, vp]
    lib.csa_attend_prefill_varlen.restype = i32
    lib.csa_index_rows_fp8.argtypes = [vp, vp, ctypes.c_longlong, vp, vp]
    lib.csa_index_rows_fp8.restype = i32
    _lib = lib
    return lib


@dataclass(frozen=True)
class Layer:
    """Mirror of csa_layer.  dtype: torch.bfloat16 or torch.float32 (model dtype).  rollback: tokens csa_trim may
    rewind; the window ring then has W + rollback slots and each frontier ring frontier_slots(ratio) + rollback.
    index_fp8: the index pool holds fp8 rows, a uint8 tensor [B, cap, FP8_ROW_BYTES]."""

    dtype: torch.dtype
    H: int
    D: int
    R: int
    W: int
    ratio: int
    Hi: int
    Di: int
    topk: int
    X: int
    scale: float = 0.0
    rms_eps: float = 1e-6
    rollback: int = 0
    index_fp8: bool = False

    @property
    def ring_slots(self) -> int:
        return self.W + self.rollback

    @property
    def lanes(self) -> int:
        return 2 if self.ratio == 4 else 1

    @property
    def has_indexer(self) -> bool:
        return self.ratio == 4

    def _c(self) -> _Layer:
        code = CSA_BF16 if self.dtype == torch.bfloat16 else CSA_F32
        return _Layer(code, self.H, self.D, self.R, self.W, self.ratio, self.Hi, self.Di, self.topk, self.X,
                      float(self.scale), float(self.rms_eps), int(self.rollback), int(self.index_fp8))

    def pool_spec(self, d: int):
        """(dtype, row length) of a pool with rows of d values: fp8 index rows are FP8_ROW_BYTES bytes."""
        if self.index_fp8 and d == self.Di:
            return torch.uint8, FP8_ROW_BYTES
        return self.dtype, d


@dataclass
class Compressor:
    """Device weights of one compressor: wkv, wgate [L*d, X] model dtype; ape [ratio, L*d] fp32; norm_w [d] fp32."""

    wkv: torch.Tensor
    wgate: torch.Tensor
    ape: torch.Tensor
    norm_w: torch.Tensor
    d: int

    def _c(self) -> _Comp:
        return _Comp(_ptr(self.wkv), _ptr(self.wgate), _ptr(self.ape), _ptr(self.norm_w), self.d)


def _expect(name: str, t, dtype: torch.dtype, shape=None, optional: bool = False):
    """Raise TypeError / ValueError unless ``t`` has ``dtype`` and (when given) exactly ``shape``."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _expect_err(err):
    if err is not None:
        _expect("err", err, torch.int32)
        if err.numel() < 1:
            raise ValueError("err must hold at least one int32")


def _expect_comp(layer: "Layer", comp: "Compressor", which: str):
    L, d = layer.lanes, comp.d
    _expect(f"{which}.wkv", comp.wkv, layer.dtype, (L * d, layer.X))
    _expect(f"{which}.wgate", comp.wgate, layer.dtype, (L * d, layer.X))
    _expect(f"{which}.ape", comp.ape, torch.float32, (layer.ratio, L * d))
    _expect(f"{which}.norm_w", comp.norm_w, torch.float32, (d,))


def _expect_pool(name: str, layer: "Layer", pool, d: int, B=None, dims: int = 3):
    """pool [B, cap, row] (dims 3) or [cap, row] (dims 2) in the layer's pool format for rows of d values."""
    dt, row = layer.pool_spec(d)
    _expect(name, pool, dt)
    lead = () if B is None or dims == 2 else (B,)
    if pool.dim() != dims or pool.shape[-1] != row or tuple(pool.shape[:len(lead)]) != lead:
        want = "[cap, %d]" % row if dims == 2 else "[%s, cap, %d]" % ("B" if B is None else B, row)
        raise ValueError(f"{name}: shape {tuple(pool.shape)}, expected {want}")


def _frontier_len(layer: "Layer") -> int:
    return (2 * layer.ratio if layer.ratio == 4 else layer.ratio) + layer.rollback


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("CSA tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("CSA tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(fn: str, code: int):
    if code != 0:
        raise CSAError(fn, code)


def kernel_launches() -> int:
    """Kernels enqueued by the library so far in this process."""
    return int(load_library().csa_kernel_launches())


def advance_positions(pos, by: int = 1, stream=None):
    """pos[b] += by for every sequence (int32 device tensor), on the library's launch path."""
    _expect("pos", pos, torch.int32, (pos.numel(),) if isinstance(pos, torch.Tensor) else None)
    _check("csa_advance_positions", load_library().csa_advance_positions(_ptr(pos), pos.numel(), by,
                                                                         _stream(stream)))


def index_rows_fp8(layer: Layer, src, dst, stream=None):
    """csa_index_rows_fp8: src [..., Di] model-dtype index rows -> dst [..., FP8_ROW_BYTES] uint8 fp8 rows (same
    leading shape); the layer has index_fp8 set."""
    _expect("src", src, layer.dtype)
    if src.dim() < 1 or src.shape[-1] != layer.Di:
        raise ValueError(f"src: shape {tuple(src.shape)}, expected [..., {layer.Di}]")
    _expect("dst", dst, torch.uint8, tuple(src.shape[:-1]) + (FP8_ROW_BYTES,))
    n = src.numel() // layer.Di
    L = layer._c()
    _check("csa_index_rows_fp8", load_library().csa_index_rows_fp8(ctypes.byref(L), _ptr(src), n, _ptr(dst),
                                                                   _stream(stream)))


def frontier_slots(ratio: int) -> int:
    return load_library().csa_frontier_slots(ratio)


def trim(layer: Layer, n_back, pos, n_rows_a, n_rows_i, hw, err=None, stream=None):
    """csa_trim: rewind each sequence b by n_back[b] tokens (int32 device tensors [B]; n_rows_i None for layers
    without an indexer; hw: the high-water positions, caller-owned).  Returns the device error word tensor."""
    B = pos.numel() if isinstance(pos, torch.Tensor) else 0
    for name, t in (("n_back", n_back), ("pos", pos), ("n_rows_a", n_rows_a), ("hw", hw)):
        _expect(name, t, torch.int32, (B,))
    _expect("n_rows_i", n_rows_i, torch.int32, (B,), optional=not layer.has_indexer)
    _expect_err(err)
    err = _err(err, pos.device)
    L = layer._c()
    _check("csa_trim", load_library().csa_trim(ctypes.byref(L), B, _ptr(n_back), _ptr(pos), _ptr(n_rows_a),
                                               _ptr(n_rows_i), _ptr(hw), _ptr(err), _stream(stream)))
    return err


def workspace_size(layer: Layer, op: int, B: int, T: int, cap: int) -> int:
    n = ctypes.c_size_t(0)
    L = layer._c()
    _check("csa_workspace_size", load_library().csa_workspace_size(ctypes.byref(L), op, B, T, cap, ctypes.byref(n)))
    return int(n.value)


def _ws(layer, op, B, T, cap, ws, device):
    need = workspace_size(layer, op, B, T, cap)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return ws, ws.numel() * ws.element_size()


def _err(err, device):
    return torch.zeros(1, dtype=torch.int32, device=device) if err is None else err


def compress_append(layer: Layer, comp: Compressor, x, pos, frontier, pool, n_rows, inv_freq, ws=None, err=None,
                    stream=None):
    """csa_compress_append; x [B,T,X]; returns the device error word tensor."""
    _expect("x", x, layer.dtype)
    if x.dim() != 3 or x.shape[2] != layer.X:
        raise ValueError(f"x: shape {tuple(x.shape)}, expected [B, T, {layer.X}]")
    B, T = x.shape[0], x.shape[1]
    _expect_comp(layer, comp, "comp")
    _expect_pool("pool", layer, pool, comp.d, B)
    cap = pool.shape[1]
    _expect("pos", pos, torch.int32, (B,))
    _expect("frontier", frontier, layer.dtype, (B, _frontier_len(layer), 2 * layer.lanes * comp.d))
    _expect("n_rows", n_rows, torch.int32, (B,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect_err(err)
    ws, nb = _ws(layer, OP_COMPRESS, B, T, cap, ws, x.device)
    err = _err(err, x.device)
    L, C = layer._c(), comp._c()
    _check("csa_compress_append", load_library().csa_compress_append(
        ctypes.byref(L), ctypes.byref(C), _ptr(x), B, T, _ptr(pos), _ptr(frontier), _ptr(pool), cap, _ptr(n_rows),
        _ptr(inv_freq), _ptr(ws), nb, _ptr(err), _stream(stream)))
    return err


def compress_append_pair(layer: Layer, comp_a: Compressor, comp_i: Compressor, x, pos, frontier_a, pool_a, n_rows_a,
                         frontier_i, pool_i, n_rows_i, inv_freq, ws=None, err=None, stream=None):
    """csa_compress_append_pair (attention pool, then index pool, same tokens); returns the error word tensor."""
    _expect("x", x, layer.dtype)
    if x.dim() != 3 or x.shape[2] != layer.X:
        raise ValueError(f"x: shape {tuple(x.shape)}, expected [B, T, {layer.X}]")
    B, T = x.shape[0], x.shape[1]
    _expect_comp(layer, comp_a, "comp_a")
    _expect_comp(layer, comp_i, "comp_i")
    F = _frontier_len(layer)
    for nm, pl, fr, nr, d in (("a", pool_a, frontier_a, n_rows_a, comp_a.d), ("i", pool_i, frontier_i, n_rows_i,
                                                                               comp_i.d)):
        _expect_pool(f"pool_{nm}", layer, pl, d, B)
        _expect(f"frontier_{nm}", fr, layer.dtype, (B, F, 2 * layer.lanes * d))
        _expect(f"n_rows_{nm}", nr, torch.int32, (B,))
    _expect("pos", pos, torch.int32, (B,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect_err(err)
    cap_a, cap_i = pool_a.shape[1], pool_i.shape[1]
    ws, nb = _ws(layer, OP_COMPRESS_PAIR, B, T, max(cap_a, cap_i), ws, x.device)
    err = _err(err, x.device)
    L, Ca, Ci = layer._c(), comp_a._c(), comp_i._c()
    _check("csa_compress_append_pair", load_library().csa_compress_append_pair(
        ctypes.byref(L), ctypes.byref(Ca), ctypes.byref(Ci), _ptr(x), B, T, _ptr(pos), _ptr(frontier_a),
        _ptr(pool_a), cap_a, _ptr(n_rows_a), _ptr(frontier_i), _ptr(pool_i), cap_i, _ptr(n_rows_i), _ptr(inv_freq),
        _ptr(ws), nb, _ptr(err), _stream(stream)))
    return err


def _expect_index(layer: Layer, iq, iw, ikeys, n_rows, pos, inv_freq, sel, n_sel, err):
    _expect("iq", iq, layer.dtype)
    if iq.dim() != 3 or iq.shape[1:] != (layer.Hi, layer.Di):
        raise ValueError(f"iq: shape {tuple(iq.shape)}, expected [B, {layer.Hi}, {layer.Di}]")
    B = iq.shape[0]
    _expect("iw", iw, layer.dtype, (B, layer.Hi))
    _expect_pool("ikeys", layer, ikeys, layer.Di, B)
    _expect("n_rows", n_rows, torch.int32, (B,))
    _expect("pos", pos, torch.int32, (B,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect("sel", sel, torch.int32, (B, layer.topk))
    _expect("n_sel", n_sel, torch.int32, (B,))
    _expect_err(err)


def index_topk(layer: Layer, iq, iw, ikeys, n_rows, pos, inv_freq, sel, n_sel, ws=None, err=None, stream=None):
    _expect_index(layer, iq, iw, ikeys, n_rows, pos, inv_freq, sel, n_sel, err)
    B, cap = iq.shape[0], ikeys.shape[1]
    ws, nb = _ws(layer, OP_INDEX_TOPK, B, 1, cap, ws, iq.device)
    err = _err(err, iq.device)
    L = layer._c()
    _check("csa_index_topk", load_library().csa_index_topk(
        ctypes.byref(L), _ptr(iq), _ptr(iw), B, _ptr(ikeys), cap, _ptr(n_rows), _ptr(pos), _ptr(inv_freq),
        _ptr(sel), _ptr(n_sel), _ptr(ws), nb, _ptr(err), _stream(stream)))
    return err


def index_topk_overlapped(layer: Layer, iq, iw, ikeys, n_rows, pos, inv_freq, sel, n_sel, pool_ready=None, ws=None,
                          err=None, stream=None):
    """csa_index_topk_overlapped: the scan of the rows complete before the token is enqueued at once; the
    rest waits for `pool_ready` (a torch.cuda.Event recorded after the index pool's compress call)."""
    _expect_index(layer, iq, iw, ikeys, n_rows, pos, inv_freq, sel, n_sel, err)
    B, cap = iq.shape[0], ikeys.shape[1]
    ws, nb = _ws(layer, OP_INDEX_TOPK, B, 1, cap, ws, iq.device)
    err = _err(err, iq.device)
    L = layer._c()
    ev = pool_ready.cuda_event if pool_ready is not None else None
    _check("csa_index_topk_overlapped", load_library().csa_index_topk_overlapped(
        ctypes.byref(L), _ptr(iq), _ptr(iw), B, _ptr(ikeys), cap, _ptr(n_rows), _ptr(pos), _ptr(inv_freq),
        _ptr(sel), _ptr(n_sel), _ptr(ws), nb, _ptr(err), _stream(stream), ev))
    return err


def index_topk_static(layer: Layer, iq, iw, ikeys, n_rows, pos, inv_freq, sel, n_sel, err=None, stream=None):
    """csa_index_topk_static: the decode indexer with the library's own fixed scratch array (no workspace)."""
    _expect_index(layer, iq, iw, ikeys, n_rows, pos, inv_freq, sel, n_sel, err)
    B, cap = iq.shape[0], ikeys.shape[1]
    err = _err(err, iq.device)
    L = layer._c()
    _check("csa_index_topk_static", load_library().csa_index_topk_static(
        ctypes.byref(L), _ptr(iq), _ptr(iw), B, _ptr(ikeys), cap, _ptr(n_rows), _ptr(pos), _ptr(inv_freq),
        _ptr(sel), _ptr(n_sel), _ptr(err), _stream(stream)))
    return err


def static_scratch_bytes() -> int:
    return int(load_library().csa_static_scratch_bytes())


def attend_decode(layer: Layer, q, kv_new, sink, window, pool, n_rows, sel, n_sel, pos, inv_freq, out, ws=None,
                  err=None, stream=None):
    _expect("q", q, layer.dtype)
    if q.dim() != 3 or q.shape[1:] != (layer.H, layer.D):
        raise ValueError(f"q: shape {tuple(q.shape)}, expected [B, {layer.H}, {layer.D}]")
    B = q.shape[0]
    _expect("kv_new", kv_new, layer.dtype, (B, layer.D))
    _expect("sink", sink, torch.float32, (layer.H,))
    _expect("window", window, layer.dtype, (B, layer.ring_slots, layer.D))
    _expect("pool", pool, layer.dtype)
    if pool.dim() != 3 or pool.shape[0] != B or pool.shape[2] != layer.D:
        raise ValueError(f"pool: shape {tuple(pool.shape)}, expected [{B}, cap, {layer.D}]")
    _expect("n_rows", n_rows, torch.int32, (B,))
    _expect("sel", sel, torch.int32, (B, layer.topk), optional=True)
    _expect("n_sel", n_sel, torch.int32, (B,), optional=sel is None)
    _expect("pos", pos, torch.int32, (B,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect("out", out, layer.dtype, (B, layer.H, layer.D))
    _expect_err(err)
    cap = pool.shape[1]
    ws, nb = _ws(layer, OP_ATTEND_DECODE, B, 1, cap, ws, q.device)
    err = _err(err, q.device)
    L = layer._c()
    _check("csa_attend_decode", load_library().csa_attend_decode(
        ctypes.byref(L), _ptr(q), _ptr(kv_new), _ptr(sink), B, _ptr(window), _ptr(pool), cap, _ptr(n_rows),
        _ptr(sel), _ptr(n_sel), _ptr(pos), _ptr(inv_freq), _ptr(out), _ptr(ws), nb, _ptr(err), _stream(stream)))
    return err


def attend_prefill_chunk(layer: Layer, q, kv_new, iq, iw, sink, pos0: int, window, pool, ikeys, n_rows, inv_freq,
                         out, sel_out=None, ws=None, err=None, stream=None):
    _expect("q", q, layer.dtype)
    if q.dim() != 3 or q.shape[1:] != (layer.H, layer.D):
        raise ValueError(f"q: shape {tuple(q.shape)}, expected [T, {layer.H}, {layer.D}]")
    T = q.shape[0]
    _expect("kv_new", kv_new, layer.dtype, (T, layer.D))
    if layer.has_indexer:
        _expect("iq", iq, layer.dtype, (T, layer.Hi, layer.Di))
        _expect("iw", iw, layer.dtype, (T, layer.Hi))
        _expect_pool("ikeys", layer, ikeys, layer.Di, dims=2)
    _expect("sink", sink, torch.float32, (layer.H,))
    _expect("window", window, layer.dtype, (layer.ring_slots, layer.D))
    _expect("pool", pool, layer.dtype)
    if pool.dim() != 2 or pool.shape[1] != layer.D:
        raise ValueError(f"pool: shape {tuple(pool.shape)}, expected [cap, {layer.D}]")
    _expect("n_rows", n_rows, torch.int32, (1,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect("out", out, layer.dtype, (T, layer.H, layer.D))
    _expect("sel_out", sel_out, torch.int32, (T, layer.topk), optional=True)
    _expect_err(err)
    cap = pool.shape[-2]
    ws, nb = _ws(layer, OP_ATTEND_PREFILL, 1, T, cap, ws, q.device)
    err = _err(err, q.device)
    L = layer._c()
    _check("csa_attend_prefill_chunk", load_library().csa_attend_prefill_chunk(
        ctypes.byref(L), _ptr(q), _ptr(kv_new), _ptr(iq), _ptr(iw), _ptr(sink), T, int(pos0), _ptr(window),
        _ptr(pool), _ptr(ikeys), cap, _ptr(n_rows), _ptr(inv_freq), _ptr(out), _ptr(sel_out), _ptr(ws), nb,
        _ptr(err), _stream(stream)))
    return err


def _expect_varlen(cu_seqlens, B: int, N: int, T_max: int):
    _expect("cu_seqlens", cu_seqlens, torch.int32, (B + 1,))
    if not 1 <= int(T_max) <= N:
        raise ValueError(f"T_max = {T_max}: expected 1 <= T_max <= N = {N}")


def compress_append_varlen(layer: Layer, comp: Compressor, x, cu_seqlens, T_max: int, pos, frontier, pool, n_rows,
                           inv_freq, ws=None, err=None, stream=None):
    """csa_compress_append_varlen; x [N, X] packs B chunks, sequence b's rows cu_seqlens[b] .. cu_seqlens[b+1]-1
    (device int32 [B+1]); T_max (host) bounds every chunk's length."""
    _expect("x", x, layer.dtype)
    if x.dim() != 2 or x.shape[1] != layer.X:
        raise ValueError(f"x: shape {tuple(x.shape)}, expected [N, {layer.X}]")
    N = x.shape[0]
    _expect_pool("pool", layer, pool, comp.d)
    B, cap = pool.shape[0], pool.shape[1]
    _expect_varlen(cu_seqlens, B, N, T_max)
    _expect_comp(layer, comp, "comp")
    _expect("pos", pos, torch.int32, (B,))
    _expect("frontier", frontier, layer.dtype, (B, _frontier_len(layer), 2 * layer.lanes * comp.d))
    _expect("n_rows", n_rows, torch.int32, (B,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect_err(err)
    ws, nb = _ws(layer, OP_COMPRESS_VARLEN, B, N, cap, ws, x.device)
    err = _err(err, x.device)
    L, C = layer._c(), comp._c()
    _check("csa_compress_append_varlen", load_library().csa_compress_append_varlen(
        ctypes.byref(L), ctypes.byref(C), _ptr(x), B, _ptr(cu_seqlens), N, int(T_max), _ptr(pos), _ptr(frontier),
        _ptr(pool), cap, _ptr(n_rows), _ptr(inv_freq), _ptr(ws), nb, _ptr(err), _stream(stream)))
    return err


def attend_prefill_varlen(layer: Layer, q, kv_new, iq, iw, sink, cu_seqlens, T_max: int, pos, window, pool, ikeys,
                          n_rows, inv_freq, out, sel_out=None, ws=None, err=None, stream=None):
    """csa_attend_prefill_varlen; q [N, H, D], kv_new [N, D], iq [N, Hi, Di], iw [N, Hi], out [N, H, D] pack B
    chunks (rows cu_seqlens[b] .. cu_seqlens[b+1]-1 at positions pos[b] ..); window [B, W+rollback, D], pool
    [B, cap, D], ikeys [B, cap, Di], n_rows [B]."""
    _expect("q", q, layer.dtype)
    if q.dim() != 3 or q.shape[1:] != (layer.H, layer.D):
        raise ValueError(f"q: shape {tuple(q.shape)}, expected [N, {layer.H}, {layer.D}]")
    N = q.shape[0]
    _expect("pool", pool, layer.dtype)
    if pool.dim() != 3 or pool.shape[2] != layer.D:
        raise ValueError(f"pool: shape {tuple(pool.shape)}, expected [B, cap, {layer.D}]")
    B, cap = pool.shape[0], pool.shape[1]
    _expect_varlen(cu_seqlens, B, N, T_max)
    _expect("kv_new", kv_new, layer.dtype, (N, layer.D))
    if layer.has_indexer:
        _expect("iq", iq, layer.dtype, (N, layer.Hi, layer.Di))
        _expect("iw", iw, layer.dtype, (N, layer.Hi))
        _expect_pool("ikeys", layer, ikeys, layer.Di, B)
        if ikeys.shape[1] != cap:
            raise ValueError(f"ikeys: shape {tuple(ikeys.shape)}, expected [{B}, {cap}, {layer.pool_spec(layer.Di)[1]}]")
    _expect("sink", sink, torch.float32, (layer.H,))
    _expect("pos", pos, torch.int32, (B,))
    _expect("window", window, layer.dtype, (B, layer.ring_slots, layer.D))
    _expect("n_rows", n_rows, torch.int32, (B,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect("out", out, layer.dtype, (N, layer.H, layer.D))
    _expect("sel_out", sel_out, torch.int32, (N, layer.topk), optional=True)
    _expect_err(err)
    ws, nb = _ws(layer, OP_ATTEND_PREFILL_VARLEN, B, N, cap, ws, q.device)
    err = _err(err, q.device)
    L = layer._c()
    _check("csa_attend_prefill_varlen", load_library().csa_attend_prefill_varlen(
        ctypes.byref(L), _ptr(q), _ptr(kv_new), _ptr(iq), _ptr(iw), _ptr(sink), B, _ptr(cu_seqlens), N, int(T_max),
        _ptr(pos), _ptr(window), _ptr(pool), _ptr(ikeys), cap, _ptr(n_rows), _ptr(inv_freq), _ptr(out), _ptr(sel_out),
        _ptr(ws), nb, _ptr(err), _stream(stream)))
    return err


def index_topk_verify(layer: Layer, iq, iw, ikeys, n_rows, pos, inv_freq, sel, n_sel, ws=None, err=None,
                      stream=None):
    """csa_index_topk_verify: iq [B, T, Hi, Di], iw [B, T, Hi]; sel [B, T, topk], n_sel [B, T]; pos [B] is the
    position of each block's first token."""
    _expect("iq", iq, layer.dtype)
    if iq.dim() != 4 or iq.shape[2:] != (layer.Hi, layer.Di):
        raise ValueError(f"iq: shape {tuple(iq.shape)}, expected [B, T, {layer.Hi}, {layer.Di}]")
    B, T = iq.shape[0], iq.shape[1]
    _expect("iw", iw, layer.dtype, (B, T, layer.Hi))
    _expect_pool("ikeys", layer, ikeys, layer.Di, B)
    _expect("n_rows", n_rows, torch.int32, (B,))
    _expect("pos", pos, torch.int32, (B,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect("sel", sel, torch.int32, (B, T, layer.topk))
    _expect("n_sel", n_sel, torch.int32, (B, T))
    _expect_err(err)
    cap = ikeys.shape[1]
    ws, nb = _ws(layer, OP_INDEX_TOPK, B * T, 1, cap, ws, iq.device)
    err = _err(err, iq.device)
    L = layer._c()
    _check("csa_index_topk_verify", load_library().csa_index_topk_verify(
        ctypes.byref(L), _ptr(iq), _ptr(iw), B, T, _ptr(ikeys), cap, _ptr(n_rows), _ptr(pos), _ptr(inv_freq),
        _ptr(sel), _ptr(n_sel), _ptr(ws), nb, _ptr(err), _stream(stream)))
    return err


def attend_verify(layer: Layer, q, kv_new, sink, window, pool, n_rows, sel, n_sel, pos, inv_freq, out, ws=None,
                  err=None, stream=None):
    """csa_attend_verify: q [B, T, H, D], kv_new [B, T, D], out [B, T, H, D]; the block's tokens are written to the
    window ring first (the layer needs rollback >= T - 1)."""
    _expect("q", q, layer.dtype)
    if q.dim() != 4 or q.shape[2:] != (layer.H, layer.D):
        raise ValueError(f"q: shape {tuple(q.shape)}, expected [B, T, {layer.H}, {layer.D}]")
    B, T = q.shape[0], q.shape[1]
    _expect("kv_new", kv_new, layer.dtype, (B, T, layer.D))
    _expect("sink", sink, torch.float32, (layer.H,))
    _expect("window", window, layer.dtype, (B, layer.ring_slots, layer.D))
    _expect("pool", pool, layer.dtype)
    if pool.dim() != 3 or pool.shape[0] != B or pool.shape[2] != layer.D:
        raise ValueError(f"pool: shape {tuple(pool.shape)}, expected [{B}, cap, {layer.D}]")
    _expect("n_rows", n_rows, torch.int32, (B,))
    _expect("sel", sel, torch.int32, (B, T, layer.topk))
    _expect("n_sel", n_sel, torch.int32, (B, T))
    _expect("pos", pos, torch.int32, (B,))
    _expect("inv_freq", inv_freq, torch.float32, (layer.R // 2,))
    _expect("out", out, layer.dtype, (B, T, layer.H, layer.D))
    _expect_err(err)
    cap = pool.shape[1]
    ws, nb = _ws(layer, OP_ATTEND_DECODE, B * T, 1, cap, ws, q.device)
    err = _err(err, q.device)
    L = layer._c()
    _check("csa_attend_verify", load_library().csa_attend_verify(
        ctypes.byref(L), _ptr(q), _ptr(kv_new), _ptr(sink), B, T, _ptr(window), _ptr(pool), cap, _ptr(n_rows),
        _ptr(sel), _ptr(n_sel), _ptr(pos), _ptr(inv_freq), _ptr(out), _ptr(ws), nb, _ptr(err), _stream(stream)))
    return err
