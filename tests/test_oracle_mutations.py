"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in the oracle (on the CPU, by patching
a function of ``oracle.csa_oracle``) and runs every pin in
``tests/test_oracle_pins.py``; at least one pin must fail.  The mistakes follow
the bug classes the pages report their own suites catching ("DeepSeek-V4-Flash:
native deepseek_v4 AR backend", MTPLX #216, "Verification": off-by-one window
keep, stale frontiers, wrong tie-break, ...; "feat: add DeepSeek-V4 (Pro/Flash)
model support", mlx-lm #1189: un-roped pool rows, a mask that blocks the pool,
sigmoid/mean in the indexer, a dropped chunk tail, a reset absolute position;
deepseek-v41-mlx README "Validation": broken inverse rope, zeroed sinks), plus
sign, index and operand slips.
"""
import inspect

import numpy as np
import pytest

from oracle import csa_oracle as O
from tests import test_oracle_pins as pins

_orig = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argname, values = params[0].args
            names = [a.strip() for a in argname.split(",")]
            for v in values:
                kw = dict(zip(names, v)) if len(names) > 1 else {names[0]: v}
                out.append((f"{name}[{v}]", fn, kw))
        else:
            out.append((name, fn, {}))
    return out


PINS = _pin_functions()


# ---------------------------------------------------------------- mutated functions

def m_window_keep_one_more(layer, p):
    return range(max(0, p - layer.W), p + 1)


def m_window_keep_one_less(layer, p):
    return range(max(0, p - layer.W + 2), p + 1)


def m_window_excludes_self(layer, p):
    return range(max(0, p - layer.W), p)


def m_stale_frontier(layer, comp, j, tok):
    """No previous-window carry: row j pools only its own window."""
    r, d = layer.ratio, comp.d
    kvs, ss = [], []
    for t in range(j * r, (j + 1) * r):
        kv, g = tok[t]
        kvs.append(kv[d:] if layer.lanes == 2 else kv)
        ss.append((g[d:] + comp.ape[t % r, d:]) if layer.lanes == 2 else g + comp.ape[t % r])
    return np.stack(kvs), np.stack(ss)


def m_lanes_swapped(layer, comp, j, tok):
    r, d = layer.ratio, comp.d
    if layer.lanes == 1:
        return _orig["window_entries"](layer, comp, j, tok)
    kvs, ss = [], []
    for t in range(max(0, (j - 1) * r), j * r):
        kv, g = tok[t]
        kvs.append(kv[d:])
        ss.append(g[d:] + comp.ape[t % r, d:])
    for t in range(j * r, (j + 1) * r):
        kv, g = tok[t]
        kvs.append(kv[:d])
        ss.append(g[:d] + comp.ape[t % r, :d])
    return np.stack(kvs), np.stack(ss)


def m_ape_index_shift(layer, comp, j, tok):
    """APE indexed from the window's last token instead of its first."""
    shifted = O.Compressor(wkv=comp.wkv, wgate=comp.wgate, ape=np.roll(comp.ape, 1, axis=0),
                           norm_w=comp.norm_w, d=comp.d)
    return _orig["window_entries"](layer, shifted, j, tok)


def m_ape_ignored(layer, comp, j, tok):
    z = O.Compressor(wkv=comp.wkv, wgate=comp.wgate, ape=np.zeros_like(comp.ape), norm_w=comp.norm_w, d=comp.d)
    return _orig["window_entries"](layer, z, j, tok)


def m_pool_weights_no_normalise(s):
    s = np.asarray(s, dtype=np.float64)
    return np.exp(s - s.max(axis=0, keepdims=True))


def m_pool_weights_wrong_axis(s):
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def m_row_not_roped(layer, comp, u, j, inv_freq):
    u = O.store(u, layer.dtype)
    return O.store(O.rms_norm(u, comp.norm_w, layer.rms_eps), layer.dtype)


def m_row_roped_at_j(layer, comp, u, j, inv_freq):
    u = O.store(u, layer.dtype)
    y = O.store(O.rms_norm(u, comp.norm_w, layer.rms_eps), layer.dtype)
    return O.store(O.rope(y, j, inv_freq), layer.dtype)


def m_row_not_normed(layer, comp, u, j, inv_freq):
    u = O.store(u, layer.dtype)
    return O.store(O.rope(u, j * layer.ratio, inv_freq), layer.dtype)


def m_rms_no_eps(u, w, eps):
    u = np.asarray(u, dtype=np.float64)
    return u / np.sqrt(np.mean(u * u, axis=-1, keepdims=True)) * w


def m_rms_sum_not_mean(u, w, eps):
    u = np.asarray(u, dtype=np.float64)
    return u / np.sqrt(np.sum(u * u, axis=-1, keepdims=True) + eps) * w


def m_rope_first_dims(v, p, inv_freq, inverse=False):
    v = np.asarray(v, dtype=np.float64)
    R = 2 * len(inv_freq)
    th = O.rope_angles(p, inv_freq) * (-1 if inverse else 1)
    out = v.copy()
    a, b = v[..., 0:R:2], v[..., 1:R:2]
    out[..., 0:R:2] = a * np.cos(th) - b * np.sin(th)
    out[..., 1:R:2] = a * np.sin(th) + b * np.cos(th)
    return out


def m_rope_half_split(v, p, inv_freq, inverse=False):
    v = np.asarray(v, dtype=np.float64)
    R, D = 2 * len(inv_freq), v.shape[-1]
    th = O.rope_angles(p, inv_freq) * (-1 if inverse else 1)
    out = v.copy()
    a, b = v[..., D - R:D - R // 2], v[..., D - R // 2:]
    out[..., D - R:D - R // 2] = a * np.cos(th) - b * np.sin(th)
    out[..., D - R // 2:] = a * np.sin(th) + b * np.cos(th)
    return out


def m_rope_sign(v, p, inv_freq, inverse=False):
    return _orig["rope"](v, p, inv_freq, inverse=not inverse)


def m_rope_exact_angle(v, p, inv_freq, inverse=False):
    v = np.asarray(v, dtype=np.float64)
    R, D = 2 * len(inv_freq), v.shape[-1]
    th = p * np.asarray(inv_freq, dtype=np.float64) * (-1 if inverse else 1)
    out = v.copy()
    a, b = v[..., D - R::2], v[..., D - R + 1::2]
    out[..., D - R::2] = a * np.cos(th) - b * np.sin(th)
    out[..., D - R + 1::2] = a * np.sin(th) + b * np.cos(th)
    return out


def m_no_inverse_rope(layer, o, p, inv_freq):
    return O.store(o, layer.dtype)


def m_visible_off_by_one(layer, n, p):
    return int(min(n, p // layer.ratio))


def m_visible_blocks_pool(layer, n, p):
    return 0


def m_visible_ignores_causality(layer, n, p):
    return int(n)


def m_index_sigmoid(layer, iq, iw, keys, p, inv_freq):
    return _orig["index_scores"](layer, iq, 1.0 / (1.0 + np.exp(-np.asarray(iw))), keys, p, inv_freq)


def m_index_mean_heads(layer, iq, iw, keys, p, inv_freq):
    q = O.store(O.rope(iq, p, inv_freq), layer.dtype)
    w = np.asarray(iw) * layer.Di ** -0.5 * layer.Hi ** -0.5
    return (w[:, None] * np.maximum(q @ np.asarray(keys).T, 0)).mean(axis=0)


def m_index_relu_after_weight(layer, iq, iw, keys, p, inv_freq):
    q = O.store(O.rope(iq, p, inv_freq), layer.dtype)
    w = np.asarray(iw) * layer.Di ** -0.5 * layer.Hi ** -0.5
    return np.maximum(w[:, None] * (q @ np.asarray(keys).T), 0).sum(axis=0)


def m_index_no_relu(layer, iq, iw, keys, p, inv_freq):
    q = O.store(O.rope(iq, p, inv_freq), layer.dtype)
    w = np.asarray(iw) * layer.Di ** -0.5 * layer.Hi ** -0.5
    return (w[:, None] * (q @ np.asarray(keys).T)).sum(axis=0)


def m_index_q_not_roped(layer, iq, iw, keys, p, inv_freq):
    return _orig["index_scores"](layer, iq, iw, keys, 0, inv_freq)


def m_index_scale_missing(layer, iq, iw, keys, p, inv_freq):
    return _orig["index_scores"](layer, iq, np.asarray(iw) * np.sqrt(layer.Di * layer.Hi), keys, p, inv_freq)


def m_topk_ties_high(scores, k):
    scores = np.asarray(scores, dtype=np.float64)
    n = len(scores)
    if n <= k:
        return np.arange(n)
    order = np.lexsort((-np.arange(n), -scores))
    return np.sort(order[:k])


def m_topk_smallest(scores, k):
    return _orig["topk_select"](-np.asarray(scores), k)


def m_topk_off_by_one(scores, k):
    return _orig["topk_select"](scores, k - 1) if len(scores) > k else _orig["topk_select"](scores, k)


def m_sink_in_numerator(layer, q, keys, sink):
    """The sink attends as a key whose value is the mean key (not the all-zero value)."""
    q, keys, z = np.asarray(q, float), np.asarray(keys, float), np.asarray(sink, float)
    logits = layer.softmax_scale * q @ keys.T
    m = np.maximum(z, logits.max(axis=1))
    e = np.exp(logits - m[:, None])
    zs = np.exp(z - m)
    return (e @ keys + zs[:, None] * keys.mean(axis=0)) / (zs + e.sum(axis=1))[:, None]


def m_sink_dropped(layer, q, keys, sink):
    return _orig["attend"](layer, q, keys, np.full(np.shape(sink), -np.inf))


def m_scale_missing(layer, q, keys, sink):
    L2 = O.Layer(**{**vars(layer), "scale": 1.0})
    return _orig["attend"](L2, q, keys, sink)


def m_attend_transposed_values(layer, q, keys, sink):
    q, keys, z = np.asarray(q, float), np.asarray(keys, float), np.asarray(sink, float)
    logits = layer.softmax_scale * q @ keys.T
    m = np.maximum(z, logits.max(axis=1))
    e = np.exp(logits - m[:, None])
    den = np.exp(z - m) + e.sum(axis=1)
    return (e / den[:, None]) @ keys[::-1]


def m_merge_no_rescale(partials, sink):
    z = np.asarray(sink, dtype=np.float64)
    Z = np.exp(z)
    acc = 0.0
    for m, l, a in partials:
        Z = Z + l
        acc = acc + a
    return acc / Z[:, None]


def m_compress_drop_tail(layer, comp, x, pos, frontier, pool, n_rows, inv_freq):
    """Chunk tail dropped: only whole windows of the chunk are kept (keep = (T//r)*r)."""
    x = np.asarray(x)
    T = x.shape[1]
    keep = (T // layer.ratio) * layer.ratio
    if keep == T or keep == 0:
        return _orig["compress_append"](layer, comp, x, pos, frontier, pool, n_rows, inv_freq)
    fr, pl, n, err = _orig["compress_append"](layer, comp, x[:, :keep], pos, frontier, pool, n_rows, inv_freq)
    return fr, pl, n, err


def m_compress_abs_pos_reset(layer, comp, x, pos, frontier, pool, n_rows, inv_freq):
    """The APE origin resets to the start of each call."""
    shift = -(np.asarray(pos) % layer.ratio)
    if np.all(shift == 0):
        return _orig["compress_append"](layer, comp, x, pos, frontier, pool, n_rows, inv_freq)
    rolled = O.Compressor(wkv=comp.wkv, wgate=comp.wgate, ape=np.roll(comp.ape, int(shift[0]), axis=0),
                          norm_w=comp.norm_w, d=comp.d)
    return _orig["compress_append"](layer, rolled, x, pos, frontier, pool, n_rows, inv_freq)


def m_compress_emit_late(layer, comp, x, pos, frontier, pool, n_rows, inv_freq):
    """Rows emitted one token late (when token (j+1)r arrives)."""
    fr, pl, n, err = _orig["compress_append"](layer, comp, x, pos, frontier, pool, n_rows, inv_freq)
    T = np.asarray(x).shape[1]
    for b in range(len(pos)):
        if (int(pos[b]) + T) % layer.ratio == 0 and n[b] > n_rows[b]:
            n[b] -= 1
    return fr, pl, n, err


def m_project_swapped(layer, comp, x):
    x = np.asarray(x, dtype=np.float64)
    return O.store(x @ comp.wgate.T, layer.dtype), O.store(x @ comp.wkv.T, layer.dtype)


def m_project_transposed(layer, comp, x):
    x = np.asarray(x, dtype=np.float64)
    return O.store(x @ comp.wkv, layer.dtype), O.store(x @ comp.wgate, layer.dtype)


def m_project_not_stored(layer, comp, x):
    x = np.asarray(x, dtype=np.float64)
    return x @ comp.wkv.T, x @ comp.wgate.T


def m_trim_keeps_rows(layer, st, n_back, hw):
    n_rows = np.array(st["n_rows"])
    err = _orig["trim"](layer, st, n_back, hw)
    st["n_rows"] = n_rows
    return err


def m_trim_margin_off_by_one(layer, st, n_back, hw):
    wide = O.Layer(**{**vars(layer), "rollback": layer.rollback + 1})
    return _orig["trim"](wide, st, n_back, hw)


def m_trim_forgets_high_water(layer, st, n_back, hw):
    return _orig["trim"](layer, st, n_back, np.array(st["pos"], dtype=np.int64))


def m_window_ring_mod_W(layer, q, kv_new, sink, window, pool, n_rows, sel, n_sel, pos, inv_freq):
    window = np.array(window, dtype=np.float64)
    Wr = window.shape[1]
    if Wr == layer.W:
        return _orig["attend_decode"](layer, q, kv_new, sink, window, pool, n_rows, sel, n_sel, pos, inv_freq)
    # reads and writes the ring modulo W instead of its own length
    small = window[:, :layer.W].copy()
    for b in range(window.shape[0]):
        for t in range(max(0, int(pos[b]) - layer.W), int(pos[b])):
            small[b, t % layer.W] = window[b, t % Wr]
    out, small, err = _orig["attend_decode"](layer, q, kv_new, sink, small, pool, n_rows, sel, n_sel, pos, inv_freq)
    p = int(pos[0])
    window[0, p % layer.W] = small[0, p % layer.W]
    return out, window, err


def m_consumer_reselects(layer, owner, window, step_in, sink, inv_freq, owner_sel=None):
    return _orig["consumer_decode_step"](layer, owner, window, step_in, sink, inv_freq, None)


def m_consumer_own_window_ignored(layer, owner, window, step_in, sink, inv_freq, owner_sel=None):
    return _orig["consumer_decode_step"](layer, owner, np.zeros_like(window), step_in, sink, inv_freq, owner_sel)


def m_store_noop(x, dtype):
    return np.asarray(x, dtype=np.float64)


def m_round_bf16_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    return np.ldexp(np.trunc(np.ldexp(x, 8 - e)), e - 8)


def m_e4m3_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    mags = O.e4m3_decode(np.arange(0x7F))
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, len(mags) - 1)
    lo = np.maximum(hi - 1, 0)
    code = np.where(a - mags[lo] < mags[hi] - a, lo, hi).astype(np.int64)
    return np.where(np.signbit(x), code | 0x80, code)


def m_fwht_sign_flipped(v):
    u = np.array(v, dtype=np.float32).copy()
    h = 1
    while h < u.shape[-1]:
        for i in range(u.shape[-1]):
            if i & h == 0:
                a, b = u[..., i].copy(), u[..., i + h].copy()
                u[..., i], u[..., i + h] = a + b, b - a
        h *= 2
    return u


def m_fp8_scale_240(v):
    u = O.fwht_f32(v)
    amax = np.float32(np.max(np.abs(u)))
    if amax == 0:
        return np.zeros(u.shape[-1], dtype=np.int64), np.float32(0.0)
    scale = np.float32(amax / np.float32(240.0))
    return O.e4m3_encode((u / scale).astype(np.float32)), scale


def m_fp8_scores_no_1_over_128(layer, q_codes, q_scales, iw, key_codes, key_scales):
    w = np.asarray(iw, dtype=np.float64) * (layer.Di ** -0.5) * (layer.Hi ** -0.5)
    dots = (O.e4m3_decode(q_codes) @ O.e4m3_decode(key_codes).T) * np.asarray(q_scales)[:, None] * \
        np.asarray(key_scales)[None, :]
    return (w[:, None] * np.maximum(dots, 0.0)).sum(axis=0)


MUTATIONS = {
    "e4m3 ties away from zero": ("e4m3_encode", m_e4m3_ties_away),
    "hadamard butterfly sign flipped": ("fwht_f32", m_fwht_sign_flipped),
    "fp8 scale amax / 240": ("quantize_fp8_row", m_fp8_scale_240),
    "fp8 scores without the 1/128": ("index_scores_fp8", m_fp8_scores_no_1_over_128),
    "window keeps W+1 tokens": ("window_tokens", m_window_keep_one_more),
    "window keeps W-1 tokens": ("window_tokens", m_window_keep_one_less),
    "window excludes the query's own token": ("window_tokens", m_window_excludes_self),
    "stale frontier (no previous-window carry)": ("window_entries", m_stale_frontier),
    "overlap lanes swapped": ("window_entries", m_lanes_swapped),
    "APE slot shifted": ("window_entries", m_ape_index_shift),
    "APE ignored": ("window_entries", m_ape_ignored),
    "pool weights not normalised": ("pool_weights", m_pool_weights_no_normalise),
    "pool softmax over channels": ("pool_weights", m_pool_weights_wrong_axis),
    "pool rows not roped": ("finalize_row", m_row_not_roped),
    "pool rows roped at j instead of j*ratio": ("finalize_row", m_row_roped_at_j),
    "pool rows not normed": ("finalize_row", m_row_not_normed),
    "rmsnorm without eps": ("rms_norm", m_rms_no_eps),
    "rmsnorm sum instead of mean": ("rms_norm", m_rms_sum_not_mean),
    "rope on first dims": ("rope", m_rope_first_dims),
    "rope half-split pairs": ("rope", m_rope_half_split),
    "rope angle sign flipped": ("rope", m_rope_sign),
    "rope angle in float64": ("rope", m_rope_exact_angle),
    "no inverse rope on output": ("output_rows", m_no_inverse_rope),
    "visibility off by one": ("visible_rows", m_visible_off_by_one),
    "mask blocks the pool": ("visible_rows", m_visible_blocks_pool),
    "visibility ignores causality": ("visible_rows", m_visible_ignores_causality),
    "sigmoid on indexer weights": ("index_scores", m_index_sigmoid),
    "mean over indexer heads": ("index_scores", m_index_mean_heads),
    "ReLU after weighting": ("index_scores", m_index_relu_after_weight),
    "no ReLU in indexer": ("index_scores", m_index_no_relu),
    "index query not roped": ("index_scores", m_index_q_not_roped),
    "index scale missing": ("index_scores", m_index_scale_missing),
    "top-k ties to the higher row": ("topk_select", m_topk_ties_high),
    "top-k of the smallest scores": ("topk_select", m_topk_smallest),
    "top-k keeps k-1": ("topk_select", m_topk_off_by_one),
    "sink in the numerator": ("attend", m_sink_in_numerator),
    "sink dropped": ("attend", m_sink_dropped),
    "softmax scale missing": ("attend", m_scale_missing),
    "values taken from the wrong rows": ("attend", m_attend_transposed_values),
    "merge without max rescale": ("merge_partials", m_merge_no_rescale),
    "chunk tail dropped": ("compress_append", m_compress_drop_tail),
    "absolute position reset per call": ("compress_append", m_compress_abs_pos_reset),
    "rows emitted one token late": ("compress_append", m_compress_emit_late),
    "kv/gate weights swapped": ("project", m_project_swapped),
    "projection contracts the weights' columns": ("project", m_project_transposed),
    "projections not rounded to the model dtype": ("project", m_project_not_stored),
    "trim keeps the row counts": ("trim", m_trim_keeps_rows),
    "trim margin one token too wide": ("trim", m_trim_margin_off_by_one),
    "trim forgets the high-water mark": ("trim", m_trim_forgets_high_water),
    "window ring indexed modulo W": ("attend_decode", m_window_ring_mod_W),
    "plain consumer re-selects with its own queries": ("consumer_decode_step", m_consumer_reselects),
    "consumer ignores its own window": ("consumer_decode_step", m_consumer_own_window_ignored),
    "storage rounding skipped": ("store", m_store_noop),
    "bf16 rounding truncates": ("round_bf16", m_round_bf16_truncate),
}


def _run_pins():
    failed = []
    for name, fn, kw in PINS:
        try:
            fn(**kw)
        except Exception:  # an assertion, or an error the mistake causes
            failed.append(name)
    return failed


def test_pins_pass_unmutated():
    assert _run_pins() == []


@pytest.mark.parametrize("label", sorted(MUTATIONS))
def test_mutation_is_caught(label, monkeypatch):
    attr, fn = MUTATIONS[label]
    monkeypatch.setattr(O, attr, fn)
    failed = _run_pins()
    assert failed, f"no pin catches: {label}"
