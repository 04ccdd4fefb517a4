"""Plain CPU oracle for one layer of DeepSeek-V4 Compressed Sparse Attention (CSA).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
bench's CPU-baseline leg may import this module; the product path never calls
it and shares no code with it.

It is slow and written to be checked by eye: float64 arithmetic, numpy library
primitives (matmul, sort, exp) as single steps, loops over sequences, tokens and
queries in the order the method defines them.  The only deliberate precision
loss is the storage rounding the pages fix: activations, caches and outputs are
held in the model dtype (bf16, or fp32 for the tiny case) while pooling, softmax
and accumulation run at full precision (MTPLX #216 "DeepSeek-V4-Flash: native
deepseek_v4 AR backend", "Decode path", on bf16 activation storage: rotary rotates in fp32 and copies back at the model dtype; the
compressor pools in fp32 and casts the row back before the norm; the sparse
attention kernel is bf16 in/out with fp32 accumulation).  Rounding happens at
exactly these points:

  * the compressor's kv and gate projections,
  * the pooled row before the norm, the norm output and the roped row,
  * the roped q, index-q and window rows,
  * the attention output before and after its inverse rotation.

Page citations use the page title and the post/section on it:
  [MTPLX#216]  "DeepSeek-V4-Flash: native deepseek_v4 AR backend"
  [mlx-lm#1189] "feat: add DeepSeek-V4 (Pro/Flash) model support"
  [v41-mlx]    "deepseek-v41-mlx" README

Readings where the pages are silent (each also listed with the design notes):
  R1  overlap lanes: rows of the previous window use lane 0 (first d channels of
      kv, gate and APE), rows of the current window use lane 1 (last d).
  R2  a ratio-4 layer emits row j once token (j+1)*4-1 arrives; row 0 has no
      previous window (its lane-0 entries are absent), so n = floor(tokens/4).
  R3  softmax scale D^-1/2; RMSNorm eps 1e-6.
  R4  window keys are the tokens t in [p-W+1, p], the query's own token included.
  R5  window and compressed keys are attended together, duplicates kept.
  R6  top-k orders by (score descending, row ascending); -0.0 == +0.0.
  R7  the indexer runs only when more than topk rows are visible; otherwise all
      visible rows are attended (same result).
  R8  the rotation angle is the fp32 product of the position and the fp32
      frequency table (both sides compute it identically); cos/sin in float64.
  R9  the attention output is rounded to the model dtype, rotated back, and
      rounded again (rotary copies back at the model dtype).
  R10 a compress call whose sequence state is inconsistent (n_rows !=
      floor(pos/ratio)), or that would emit a row at or beyond the pool
      capacity, changes nothing for that sequence and raises an error bit.
  R15 rollback: the window ring and the frontier rings may hold extra slots
      (the rollback margin, whose frontier slots are the journal of projected
      rows); every ring is indexed modulo its own length, so extra slots change
      no result.  A trim back to position p' is refused unless p' >= 0 and
      p' >= (the highest position the sequence reached) - rollback.
  R16 cross-layer sharing (V4.1): a layer without a compressor keeps its own
      window ring and attends to the most recent owner's compressed rows,
      through its own top-k over the owner's index keys (index-source layers)
      or through the owner's selection of the same step (the other layers).
  R19 fp8 index keys (the optional key format): the pages name a Hadamard
      rotation of the indexer's activations and an fp4 activation simulation
      without fixing a format ([mlx-lm#1189], the indexer thread).  This build's
      format: every index row and every index-query head (128 values, already
      in the model dtype) is rotated by the unnormalised 128-point Walsh-Hadamard
      transform (butterflies of spans 1, 2, .., 64 in fp32), scaled by
      amax / 448 (fp32) and rounded to E4M3 (nearest even, saturating at 448);
      a row keeps its 128 codes and its fp32 scale.  The score is the bf16
      definition with the dot product taken on the decoded values and divided by
      128 (H H^T = 128 I, so the rotation cancels).  The codes are integers
      decided in fp32 on both sides, in the same operation order.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# error bits, the same meaning as the library's device error word
ERR_CAPACITY = 1
ERR_STATE = 2
ERR_RANGE = 4
ERR_ROLLBACK = 8


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------

def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), once.

    bf16 keeps 8 significant bits and fp32's exponent range.  Writing
    x = m * 2^e with 0.5 <= |m| < 1, the representable neighbours are the
    multiples of 2^(e-8); below the smallest normal (2^-126) the spacing stays
    2^-133 (subnormals).
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    return np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)


def round_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def store(x, dtype: str) -> np.ndarray:
    """Value of ``x`` once written to a buffer of the model dtype."""
    return round_bf16(x) if dtype == "bf16" else round_f32(x)


# --------------------------------------------------------------------------
# layer description
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Layer:
    dtype: str
    H: int
    D: int
    R: int
    W: int
    ratio: int
    Hi: int
    Di: int
    topk: int
    X: int
    scale: float | None = None  # default D^-1/2 (R3)
    rms_eps: float = 1e-6  # (R3)
    rollback: int = 0  # tokens trim() may rewind (R15)

    @property
    def lanes(self) -> int:
        """Ratio-4 layers pool overlapping windows through two lanes
        ([mlx-lm#1189], Thump604's fixes: the overlap compressor's ape is [4, 1024]
        and wkv/wgate [1024, 4096], two lanes of 512); ratio-128 layers use one."""
        return 2 if self.ratio == 4 else 1

    @property
    def frontier_slots(self) -> int:
        """Tokens the frontier ring keeps: the current and the previous window
        when windows overlap, the current window otherwise."""
        return 2 * self.ratio if self.lanes == 2 else self.ratio

    @property
    def has_indexer(self) -> bool:
        """Only ratio-4 layers carry the top-k indexer ([mlx-lm#1189], machiabeli's
        v0.2 indexer top-k post: the indexer runs on the ratio-4 layers)."""
        return self.ratio == 4

    @property
    def softmax_scale(self) -> float:
        return float(self.D) ** -0.5 if self.scale is None else float(self.scale)


@dataclass
class Compressor:
    wkv: np.ndarray  # [L*d, X] model-dtype values
    wgate: np.ndarray  # [L*d, X]
    ape: np.ndarray  # [ratio, L*d] fp32 values
    norm_w: np.ndarray  # [d] fp32 values
    d: int


# --------------------------------------------------------------------------
# RoPE and RMSNorm
# --------------------------------------------------------------------------

def rope_angles(p, inv_freq) -> np.ndarray:
    """theta_i = p * inv_freq[i], one fp32 multiply (R8; [mlx-lm#1189] stepnoy's
    apply_positions: positions cast to float32 times inv_freq)."""
    return (np.float32(p) * np.asarray(inv_freq, dtype=np.float32)).astype(np.float64)


def rope(v, p, inv_freq, inverse: bool = False) -> np.ndarray:
    """Rotate the LAST 2*len(inv_freq) dims of v (any leading shape) at position p.

    Interleaved pairs: dims (D-R+2i, D-R+2i+1) rotate by theta_i
    ([mlx-lm#1189] stepnoy: the rotation acts on the trailing rope dims; pairs
    x0 = rot[..., 0], x1 = rot[..., 1] -> (x0 cos - x1 sin, x0 sin + x1 cos)).
    ``inverse`` rotates by -theta (the output rotation, [mlx-lm#1189] Thump604:
    the rope dims of the attention output are rotated back).
    """
    v = np.asarray(v, dtype=np.float64)
    R = 2 * len(inv_freq)
    D = v.shape[-1]
    th = rope_angles(p, inv_freq)
    if inverse:
        th = -th
    c, s = np.cos(th), np.sin(th)
    out = v.copy()
    a = v[..., D - R::2]
    b = v[..., D - R + 1::2]
    out[..., D - R::2] = a * c - b * s
    out[..., D - R + 1::2] = a * s + b * c
    return out


def rms_norm(u, w, eps) -> np.ndarray:
    """y = u / sqrt(mean(u^2) + eps) * w over the last axis."""
    u = np.asarray(u, dtype=np.float64)
    return u / np.sqrt(np.mean(u * u, axis=-1, keepdims=True) + eps) * np.asarray(w, dtype=np.float64)


# --------------------------------------------------------------------------
# compressor (gated pooling)
# --------------------------------------------------------------------------

def project(layer: Layer, comp: Compressor, x) -> tuple[np.ndarray, np.ndarray]:
    """kv_t = Wkv x_t and g_t = Wgate x_t, stored at the model dtype.  x [..., X]."""
    x = np.asarray(x, dtype=np.float64)
    kv = store(x @ comp.wkv.T, layer.dtype)
    g = store(x @ comp.wgate.T, layer.dtype)
    return kv, g


def pool_weights(s) -> np.ndarray:
    """Per-channel softmax over the window's entries (axis 0).  s [E, d]."""
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - s.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


def window_entries(layer: Layer, comp: Compressor, j: int, tok: dict):
    """The (kv, score) entries pooled into compressed row j.

    ``tok`` maps absolute token index -> (kv [L*d], g [L*d]).  The score of an
    entry is its gate plus the absolute position embedding of the token's slot
    in its window, ape[t mod ratio] ([MTPLX#216] "What V4 adds": learned gated
    pooling; [mlx-lm#1189] OmarB97/aidiffuser: rows carry the previous window
    for the ratio-4 overlap transform).
    Ratio 4 (R1): tokens of window j-1 through lane 0 and tokens of window j
    through lane 1; window -1 does not exist, so row 0 pools 4 entries.
    Ratio 128: the 128 tokens of window j through the single lane.
    """
    r, d = layer.ratio, comp.d
    kvs, ss = [], []
    if layer.lanes == 2:
        for t in range((j - 1) * r, j * r):
            if t < 0:
                continue
            kv, g = tok[t]
            kvs.append(kv[:d])
            ss.append(g[:d] + comp.ape[t % r, :d])
        for t in range(j * r, (j + 1) * r):
            kv, g = tok[t]
            kvs.append(kv[d:])
            ss.append(g[d:] + comp.ape[t % r, d:])
    else:
        for t in range(j * r, (j + 1) * r):
            kv, g = tok[t]
            kvs.append(kv)
            ss.append(g + comp.ape[t % r])
    return np.stack(kvs), np.stack(ss)


def finalize_row(layer: Layer, comp: Compressor, u, j: int, inv_freq) -> np.ndarray:
    """Pooled row -> model dtype -> RMSNorm -> model dtype -> RoPE at j*ratio -> model dtype.

    ([MTPLX#216] "Decode path": the compressor pools in fp32 and casts the row
    back before the norm; [mlx-lm#1189] OmarB97's RoPE fixes: a pool row is
    rotated when it is emitted, at the position its window starts, 0, r, 2r, ...)
    """
    u = store(u, layer.dtype)
    y = store(rms_norm(u, comp.norm_w, layer.rms_eps), layer.dtype)
    return store(rope(y, j * layer.ratio, inv_freq), layer.dtype)


def compressor_row(layer: Layer, comp: Compressor, j: int, tok: dict, inv_freq) -> np.ndarray:
    kv, s = window_entries(layer, comp, j, tok)
    u = (pool_weights(s) * kv).sum(axis=0)
    return finalize_row(layer, comp, u, j, inv_freq)


def compress_append(layer: Layer, comp: Compressor, x, pos, frontier, pool, n_rows, inv_freq, proj=None):
    """Append T tokens per sequence to one compressed pool (attention or index).

    x [B,T,X]; pos [B] position of x[:,0]; frontier [B,F,2*L*d] ring of the
    projected (kv | gate) rows of the last F tokens, slot t mod F; pool
    [B,cap,d]; n_rows [B].  Row j is emitted when token (j+1)*ratio-1 arrives
    (R2), so rows built one token at a time equal rows built from a chunk
    ([mlx-lm#1189] stepnoy "Fix" 3: the chunk tail is buffered and replayed, the
    absolute position accumulates).  F is the frontier ring's own length (the
    base slots, plus the rollback journal when the layer keeps one, R15).  ``proj`` = (kv [B,T,L*d], g [B,T,L*d])
    optionally supplies the stored projections of the new tokens instead of
    computing them from x (so pooling can be checked on given inputs).
    Returns (frontier, pool, n_rows, err).
    """
    x = np.asarray(x, dtype=np.float64)
    frontier = np.array(frontier, dtype=np.float64)
    pool = np.array(pool, dtype=np.float64)
    n_rows = np.array(n_rows, dtype=np.int64)
    B, T, _ = x.shape
    r, F, cap = layer.ratio, frontier.shape[1], pool.shape[1]
    Ld = layer.lanes * comp.d
    if proj is None:
        kv_all, g_all = project(layer, comp, x)
    else:
        kv_all, g_all = (np.asarray(a, dtype=np.float64) for a in proj)
    err = 0
    for b in range(B):
        p0 = int(pos[b])
        last_row = (p0 + T) // r - 1
        if p0 < 0 or n_rows[b] != p0 // r:
            err |= ERR_STATE
            continue
        if last_row >= cap:
            err |= ERR_CAPACITY
            continue
        tok = {}
        for t in range(max(0, p0 - F), p0):
            tok[t] = (frontier[b, t % F, :Ld], frontier[b, t % F, Ld:])
        for i in range(T):
            p = p0 + i
            tok[p] = (kv_all[b, i], g_all[b, i])
            if (p + 1) % r == 0:
                j = (p + 1) // r - 1
                pool[b, j] = compressor_row(layer, comp, j, tok, inv_freq)
                n_rows[b] = j + 1
        for t in range(max(0, p0 + T - F), p0 + T):
            frontier[b, t % F] = np.concatenate(tok[t])
    return frontier, pool, n_rows, err


# --------------------------------------------------------------------------
# indexer
# --------------------------------------------------------------------------

def visible_rows(layer: Layer, n: int, p: int) -> int:
    """Rows visible to the query at absolute position p: row j pools tokens
    [j*r, (j+1)*r - 1], so it is visible iff (j+1)*r <= p+1 ([mlx-lm#1189]
    OmarB97's fix of the compressed-row visibility mask; stepnoy's patch point 1)."""
    return int(min(n, (p + 1) // layer.ratio))


def index_scores(layer: Layer, iq, iw, keys, p, inv_freq) -> np.ndarray:
    """score_j = sum_h w_h * ReLU(RoPE(iq_h, p) . key_j), w_h = iw_h * Di^-1/2 * Hi^-1/2.

    ([mlx-lm#1189] stepnoy's patch point 3 and aidiffuser's indexer: raw
    weights_proj output with the softmax scale folded, no sigmoid, ReLU on the
    logits, summed over heads; queries roped at their absolute position.)
    iq [Hi, Di]; iw [Hi]; keys [n, Di] (already roped at j*ratio by the compressor).
    """
    q = store(rope(iq, p, inv_freq), layer.dtype)
    w = np.asarray(iw, dtype=np.float64) * (layer.Di ** -0.5) * (layer.Hi ** -0.5)
    dots = q @ np.asarray(keys, dtype=np.float64).T  # [Hi, n]
    return (w[:, None] * np.maximum(dots, 0.0)).sum(axis=0)


def topk_select(scores, k: int) -> np.ndarray:
    """Indices of the k largest scores, ties to the lower row (R6), ascending order."""
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.shape[0]
    if n <= k:
        return np.arange(n, dtype=np.int64)
    order = np.lexsort((np.arange(n), -scores))  # primary -score, secondary index
    return np.sort(order[:k])


def select_rows(layer: Layer, iq, iw, keys, n_vis: int, p: int, inv_freq):
    """Rows the query at p attends (R7): all visible rows, or the indexer's top-k."""
    if not layer.has_indexer or n_vis <= layer.topk:
        return np.arange(n_vis, dtype=np.int64), None
    s = index_scores(layer, iq, iw, keys[:n_vis], p, inv_freq)
    return topk_select(s, layer.topk), s


def index_topk(layer: Layer, iq, iw, ikeys, n_rows, pos, inv_freq):
    """Decode indexer: one query per sequence at pos[b].  Returns sel [B,topk]
    (ascending rows, -1 padding) and n_sel [B]."""
    B = len(pos)
    sel = -np.ones((B, layer.topk), dtype=np.int64)
    n_sel = np.zeros(B, dtype=np.int64)
    for b in range(B):
        p = int(pos[b])
        nv = visible_rows(layer, int(n_rows[b]), p)
        rows, _ = select_rows(layer, iq[b], iw[b], ikeys[b], nv, p, inv_freq)
        sel[b, :len(rows)] = rows
        n_sel[b] = len(rows)
    return sel, n_sel


# --------------------------------------------------------------------------
# fp8 index keys (R19)
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_decode(code) -> np.ndarray:
    """Value of E4M3 codes (OCP 8-bit floating point: sign, 4 exponent bits of bias 7, 3 mantissa bits; exponent 0
    holds the subnormals m * 2^-9; S.1111.111 is NaN, there is no infinity)."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code of each (finite) value, ties to the even code, magnitudes beyond 448 saturating to 448,
    the sign bit that of the value (-0 -> 0x80).
    Written from the format: the representable magnitudes are m * 2^-9 (m = 0..7) and (8 + m) * 2^(e-10)
    (e = 1..15, m = 0..7, except e = 15, m = 7); the code of a magnitude is its index in that increasing list,
    so the nearest one, with ties to the even index, is the nearest even-mantissa one."""
    x = np.asarray(x, dtype=np.float64)
    mags = e4m3_decode(np.arange(0x7F))  # codes 0x00 .. 0x7E: 0 .. 448, increasing
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, len(mags) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - mags[lo], mags[hi] - a
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = pick.astype(np.int64)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.int64)  # the sign is kept, zero's included


def fwht_f32(v) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform of 128 values in fp32, butterflies of span 1, 2, 4, .., 64 in that
    order, (a, b) -> (a + b, a - b) for each pair (i, i + span) with bit `span` of i clear (R19)."""
    u = np.array(v, dtype=np.float32).copy()
    n = u.shape[-1]
    h = 1
    while h < n:
        for i in range(n):
            if i & h == 0:
                a, b = u[..., i].copy(), u[..., i + h].copy()
                u[..., i] = a + b
                u[..., i + h] = a - b
        h *= 2
    return u


def quantize_fp8_row(v):
    """(codes [128], scale) of one index row or index-query head already in the model dtype (R19): fp32 rotation,
    scale = amax / 448 (fp32), codes = E4M3(u / scale); an all-zero row has scale 0 and zero codes."""
    u = fwht_f32(v)
    amax = np.float32(np.max(np.abs(u)))
    if amax == 0:
        return np.zeros(u.shape[-1], dtype=np.int64), np.float32(0.0)
    scale = np.float32(amax / np.float32(E4M3_MAX))
    return e4m3_encode((u / scale).astype(np.float32)), scale


def fp8_key_values(codes, scale) -> np.ndarray:
    """Rotated, quantised key row as float64: decoded codes times the row's scale."""
    return e4m3_decode(codes) * np.float64(scale)


def index_scores_fp8(layer: Layer, q_codes, q_scales, iw, key_codes, key_scales) -> np.ndarray:
    """score_j = sum_h w_h ReLU(s_q[h] s_k[j] (qc_h . kc_j) / 128), the bf16 definition on the rotated,
    quantised operands (R19).  q_codes [Hi, 128], q_scales [Hi]; key_codes [n, 128], key_scales [n]."""
    w = np.asarray(iw, dtype=np.float64) * (layer.Di ** -0.5) * (layer.Hi ** -0.5)
    qv = e4m3_decode(q_codes)
    kv = e4m3_decode(key_codes)
    dots = (qv @ kv.T) * np.asarray(q_scales, dtype=np.float64)[:, None] * np.asarray(key_scales,
                                                                                     dtype=np.float64)[None, :]
    return (w[:, None] * np.maximum(dots / 128.0, 0.0)).sum(axis=0)


def quantize_fp8_query(layer: Layer, iq, p, inv_freq):
    """(codes [Hi, 128], scales [Hi]) of the index query at position p: RoPE as for the bf16 scores, the model
    dtype, then quantize_fp8_row per head."""
    q = store(rope(iq, p, inv_freq), layer.dtype)
    out = [quantize_fp8_row(q[h]) for h in range(q.shape[0])]
    return np.stack([c for c, _ in out]), np.array([s for _, s in out], dtype=np.float32)


# --------------------------------------------------------------------------
# attention with sink, and the split-K merge
# --------------------------------------------------------------------------

def attend(layer: Layer, q, keys, sink) -> np.ndarray:
    """Softmax attention of H heads over one shared set of keys (K = V).

    q [H, D] (roped, model dtype); keys [N, D]; sink [H].  The sink logit z_h
    enters the softmax denominator only ([v41-mlx]: the sinks are added to the
    softmax denominator alone; [MTPLX#216] "What V4 adds": one sink logit per head):
        o_h = sum_t e^{l_ht} key_t / (e^{z_h} + sum_t e^{l_ht}),  l_ht = scale q_h . key_t
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    z = np.asarray(sink, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros_like(q)
    logits = layer.softmax_scale * (q @ keys.T)  # [H, N]
    m = np.maximum(z, logits.max(axis=1))
    e = np.exp(logits - m[:, None])
    denom = np.exp(z - m) + e.sum(axis=1)
    return (e @ keys) / denom[:, None]


def attend_partial(layer: Layer, q, keys):
    """Unnormalised partial over one key subset: (m, l, acc) per head.
    m = max logit (-inf if empty), l = sum e^{l-m}, acc = sum e^{l-m} key."""
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    H, D = q.shape
    if keys.shape[0] == 0:
        return np.full(H, -np.inf), np.zeros(H), np.zeros((H, D))
    logits = layer.softmax_scale * (q @ keys.T)
    m = logits.max(axis=1)
    e = np.exp(logits - m[:, None])
    return m, e.sum(axis=1), e @ keys


def merge_partials(partials, sink) -> np.ndarray:
    """Split-K merge of (m_s, l_s, acc_s) partials with the sink added once:
    M = max(z, max_s m_s); Z = e^{z-M} + sum_s l_s e^{m_s-M}; o = sum_s acc_s e^{m_s-M} / Z.
    (Log-sum-exp algebra; equal to attend() over the union of the subsets.)"""
    z = np.asarray(sink, dtype=np.float64)
    M = z.copy()
    for m, _, _ in partials:
        M = np.maximum(M, m)
    Z = np.exp(z - M)
    acc = 0.0
    for m, l, a in partials:
        f = np.where(np.isfinite(m), np.exp(m - M), 0.0)
        Z = Z + l * f
        acc = acc + a * f[:, None]
    return acc / Z[:, None]


def output_rows(layer: Layer, o, p, inv_freq) -> np.ndarray:
    """Attention output -> model dtype -> inverse RoPE at p -> model dtype (R9)."""
    o = store(o, layer.dtype)
    return store(rope(o, p, inv_freq, inverse=True), layer.dtype)


def window_tokens(layer: Layer, p: int) -> range:
    """Raw tokens in the sliding window of the query at p (R4)."""
    return range(max(0, p - layer.W + 1), p + 1)


def attend_decode(layer: Layer, q, kv_new, sink, window, pool, n_rows, sel, n_sel, pos, inv_freq):
    """One decode step's attention for every sequence.

    Appends RoPE(kv_new, p) to the window ring (slot p mod the ring's length:
    W, plus the rollback margin when kept, R15), then attends q roped at p over
    the selected pool rows (``sel`` None: every visible row, the ratio-128 /
    dense layers) plus the window tokens [p-W+1, p].
    Returns (out [B,H,D], window, err).  A selected index outside [0, n_rows)
    raises ERR_RANGE and is skipped.
    """
    window = np.array(window, dtype=np.float64)
    B = len(pos)
    Wr = window.shape[1]
    out = np.zeros((B, layer.H, layer.D))
    err = 0
    for b in range(B):
        p = int(pos[b])
        window[b, p % Wr] = store(rope(kv_new[b], p, inv_freq), layer.dtype)
        if sel is None:
            rows = np.arange(visible_rows(layer, int(n_rows[b]), p))
        else:
            rows = np.asarray(sel[b][: int(n_sel[b])], dtype=np.int64)
            bad = (rows < 0) | (rows >= int(n_rows[b]))
            if bad.any():
                err |= ERR_RANGE
                rows = rows[~bad]
        keys = [pool[b][rows]] + [window[b, t % Wr][None] for t in window_tokens(layer, p)]
        keys = np.concatenate(keys, axis=0)
        qr = store(rope(q[b], p, inv_freq), layer.dtype)
        out[b] = output_rows(layer, attend(layer, qr, keys, sink), p, inv_freq)
    return out, window, err


def attend_prefill_chunk(layer: Layer, q, kv_new, iq, iw, sink, pos0, window, pool, ikeys, n_rows,
                         inv_freq, queries=None):
    """Attention for a chunk of T tokens at positions pos0 .. pos0+T-1 (batch 1).

    The compressors have already consumed the whole chunk, so the pool holds
    rows emitted up to the chunk's end; each query attends only the rows
    visible to it, through its OWN top-k ([mlx-lm#1189] stepnoy's patch point
    3: each query's own top-k membership is combined with the visibility mask;
    aidiffuser: a membership scatter instead of one shared gathered set).
    Window keys older than the chunk come from the ring; chunk tokens are
    roped at their own positions.  After the chunk the ring holds its last W
    tokens (its last W + rollback when the ring keeps a rollback margin, R15).  ``queries`` optionally restricts which chunk offsets are computed
    (for sampled checks at full size); the others stay zero.
    Returns (out [T,H,D], sel [T,topk] (-1 padding), n_sel [T], window).
    """
    q = np.asarray(q, dtype=np.float64)
    T = q.shape[0]
    window = np.array(window, dtype=np.float64)
    W, Wr, k = layer.W, window.shape[0], layer.topk
    kvr = [store(rope(kv_new[i], pos0 + i, inv_freq), layer.dtype) for i in range(T)]
    out = np.zeros((T, layer.H, layer.D))
    sel = -np.ones((T, k), dtype=np.int64)
    n_sel = np.zeros(T, dtype=np.int64)
    for i in (range(T) if queries is None else queries):
        p = pos0 + i
        nv = visible_rows(layer, int(n_rows), p)
        rows, _ = select_rows(layer, iq[i] if iq is not None else None,
                              iw[i] if iw is not None else None,
                              ikeys, nv, p, inv_freq)
        if layer.has_indexer:
            sel[i, :len(rows)] = rows
            n_sel[i] = len(rows)
        win = [window[t % Wr] if t < pos0 else kvr[t - pos0] for t in window_tokens(layer, p)]
        keys = np.concatenate([pool[rows], np.stack(win)], axis=0)
        qr = store(rope(q[i], p, inv_freq), layer.dtype)
        out[i] = output_rows(layer, attend(layer, qr, keys, sink), p, inv_freq)
    for t in range(max(pos0, pos0 + T - Wr), pos0 + T):
        window[t % Wr] = kvr[t - pos0]
    return out, sel, n_sel, window


# --------------------------------------------------------------------------
# a whole decode step (for the decode == prefill equivalence)
# --------------------------------------------------------------------------

def decode_step(layer: Layer, comp_a: Compressor, comp_i: Compressor | None, st: dict, step_in, sink,
                inv_freq):
    """One token for every sequence through the four calls in order:
    compress (attention pool), compress (index pool), indexer top-k, attention.
    ``st`` holds pool, ikeys, window, front_a, front_i, n_rows, pos (updated in place;
    pos advanced by one).  Returns (out, sel, n_sel, err)."""
    x, q, kv, iq, iw = step_in
    err = 0
    n0 = st["n_rows"].copy()
    st["front_a"], st["pool"], n_a, e = compress_append(layer, comp_a, x, st["pos"], st["front_a"],
                                                        st["pool"], n0, inv_freq)
    err |= e
    if layer.has_indexer:
        st["front_i"], st["ikeys"], n_i, e = compress_append(layer, comp_i, x, st["pos"], st["front_i"],
                                                             st["ikeys"], n0, inv_freq)
        err |= e
        assert np.array_equal(n_a, n_i)  # index rows == pool rows ([mlx-lm#1189] stepnoy "Fix" 2)
        sel, n_sel = index_topk(layer, iq, iw, st["ikeys"], n_a, st["pos"], inv_freq)
    else:
        sel, n_sel = None, None
    st["n_rows"] = n_a
    out, st["window"], e = attend_decode(layer, q, kv, sink, st["window"], st["pool"], n_a, sel, n_sel,
                                         st["pos"], inv_freq)
    err |= e
    st["pos"] = np.asarray(st["pos"]) + 1
    return out, sel, n_sel, err


# --------------------------------------------------------------------------
# exact trim (speculative decoding's rejection repair)
# --------------------------------------------------------------------------

def trim(layer: Layer, st: dict, n_back, hw):
    """Rewind each sequence b by n_back[b] tokens ([MTPLX#216], the MTP /
    speculative-lane post: the cache trim rewinds every lane exactly; compressed
    rows are truncated, since each depends only on its own completed window; the
    compressor frontiers are rebuilt from a bounded journal of projected rows;
    the window keeps rollback_capacity extra rows; beyond that bound trim refuses
    rather than clamps).  With the journal and the extra window rows kept in the
    rings' rollback slots (R15) nothing is copied: the position and both row
    counts move back, and the rings and pools keep the older entries the next
    tokens need.  ``hw`` holds each sequence's highest position so far (updated
    here); a sequence whose trim is refused keeps its whole state.  Returns the
    error bits (ERR_ROLLBACK, ERR_STATE)."""
    err = 0
    pos = np.array(st["pos"], dtype=np.int64)
    n_rows = np.array(st["n_rows"], dtype=np.int64)
    for b in range(len(pos)):
        p, n = int(pos[b]), int(n_back[b])
        h = max(int(hw[b]), p)
        if p < 0 or n_rows[b] != p // layer.ratio:
            err |= ERR_STATE
            continue
        if n < 0 or p - n < 0 or p - n < h - layer.rollback:
            err |= ERR_ROLLBACK
            continue
        hw[b] = h
        pos[b] = p - n
        n_rows[b] = (p - n) // layer.ratio
    st["pos"], st["n_rows"] = pos, n_rows
    return err


# --------------------------------------------------------------------------
# cross-layer sharing (DeepSeek-V4.1)
# --------------------------------------------------------------------------

def consumer_decode_step(layer: Layer, owner: dict, window, step_in, sink, inv_freq, owner_sel=None):
    """One decode step of a layer that owns no compressor ([v41-mlx], "Cross-layer sharing": a few layers own
    the KV compressors and index keys and every other layer consumes the most recent owner's caches; the
    index-source layers score their own queries against the owner's keys).  Reading R16: such a layer keeps its
    own sliding-window ring (its own kv rows) and attends, with its own queries and sinks, to the owner's
    compressed rows: through its own top-k over the owner's index keys when it is an index-source layer
    (``owner_sel`` None), else through the owner's selection of this step (``owner_sel`` = (sel, n_sel)).  It
    writes none of the owner's state.  ``owner`` holds the owner's pool, ikeys, n_rows after this step's
    compress calls, and the step's positions.  Returns (out, sel, n_sel, window, err)."""
    x, q, kv, iq, iw = step_in
    if owner_sel is None:
        sel, n_sel = index_topk(layer, iq, iw, owner["ikeys"], owner["n_rows"], owner["pos"], inv_freq)
    else:
        sel, n_sel = owner_sel
    out, window, err = attend_decode(layer, q, kv, sink, window, owner["pool"], owner["n_rows"], sel, n_sel,
                                     owner["pos"], inv_freq)
    return out, sel, n_sel, window, err
