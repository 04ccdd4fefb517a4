"""Helpers of the GPU parity tests: device copies of the seeded inputs, library
calls through the binding, and the comparison rules.

Comparison rules (tolerances the tests use):
  * top-k sets: if the oracle's k-th and (k+1)-th scores differ by more than
    1e-3 relative, the GPU set must equal the oracle set exactly; otherwise every
    row scoring above s_k (1 + 1e-3) must be selected and none below s_k (1 - 1e-3).
  * attention outputs: the oracle recomputes attention with the GPU's selected
    rows; per (query, head) row every element must satisfy
    |gpu - oracle| <= max(TOL * max|oracle row|, one ulp of the model dtype at the
    oracle value), TOL = 2e-3 for bf16 and 1e-5 for fp32.  Both sides round the
    output to the model dtype, so an element whose exact value sits at a rounding
    boundary may land one ulp apart; that is the second term.  On the rope dims,
    which are rounded, rotated back and rounded again, two ulps of the rotated
    pair's norm are added (a flip of the partner enters through the rotation).
    Where the test also has the oracle's output before any storage rounding
    (float64 attention, rotated back), the non-rope dims must in addition lie
    within TOL * max|exact row| + half an ulp of the model dtype of that exact
    value: the GPU may lose no more than its one rounding to the model dtype plus
    TOL.  (On the rope dims the output is rounded, rotated and rounded again, R9,
    so the rounded rule above is the one that applies there.)  The worst
    max-relative errors seen per workload are collected in ``WORST`` and printed
    at the end of the session.
  * compressor projections (kv | gate of each token, fp32 accumulation on the GPU,
    float64 in the oracle, both rounded once): within one ulp of the model dtype
    plus 2^-16 of sum_k |w_k x_k| (fp32 accumulation error on cancelling sums).
  * compressed rows: the oracle pools the GPU's own projections (checked above),
    then rows must agree within 2 ulps of the model dtype per element, plus 2 ulps
    of the larger element of a rotated pair on the rope dims, plus 2^-20 of the
    row's largest element where a rotation cancels a value to near zero (bf16),
    or within 1e-5 of the row's largest element (fp32).
"""
from __future__ import annotations

import numpy as np
import torch

import csa_synth
import deepseek_v4_compressed_csa_gb300 as csa
from oracle import csa_oracle as O
from tests._common import f64

TOL = {"bf16": 2e-3, "f32": 1e-5}


def dev(t):
    return None if t is None else t.to("cuda").contiguous()


def lib_layer(cfg: csa_synth.Config) -> csa.Layer:
    return csa.Layer(dtype=cfg.storage, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi, Di=cfg.Di,
                     topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps, rollback=cfg.rollback)


def lib_comp(c: csa_synth.Compressor) -> csa.Compressor:
    return csa.Compressor(wkv=dev(c.wkv), wgate=dev(c.wgate), ape=dev(c.ape), norm_w=dev(c.norm_w), d=c.d)


class DevCache:
    def __init__(self, cache: csa_synth.Cache):
        self.pool = dev(cache.pool)
        self.ikeys = dev(cache.ikeys)
        self.window = dev(cache.window)
        self.front_attn = dev(cache.front_attn)
        self.front_index = dev(cache.front_index)
        self.n_rows = dev(cache.n_rows)
        self.pos = dev(cache.pos)


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the model dtype at |x| (bf16: 8 significant bits; fp32: 24)."""
    bits = 8 if dtype == "bf16" else 24
    _, e = np.frexp(np.abs(x))
    e = np.maximum(e, -125)
    return np.ldexp(1.0, e - bits)


# workload label -> worst max-relative output errors seen by check_rows:
#   "rounded": against the oracle's output rounded as the pages store it (all dims)
#   "exact_nonrope": against the oracle's un-rounded output, on the dims the inverse rotation leaves alone (this
#       includes the output's own rounding to the model dtype: up to 2^-8 of an element in bf16)
#   "beyond_rounding": the same, less half an ulp of each exact element: what the kernels lose beyond that rounding
#   "rows": (query, head) rows checked
WORST: dict[str, dict] = {}


def _record(label, key, value, rows):
    w = WORST.setdefault(label, {"rounded": 0.0, "exact_nonrope": 0.0, "beyond_rounding": 0.0, "rows": 0})
    w[key] = max(w[key], value)
    if key == "rounded":
        w["rows"] += rows


def exact_output(o, p: int, inv_freq) -> np.ndarray:
    """The oracle's attention output before any storage rounding: float64 o (from O.attend) rotated back by
    -theta(p) on the rope dims."""
    return O.rope(o, p, inv_freq, inverse=True)


def check_rows(gpu, ref, dtype: str, what: str = "output", R: int = 0, exact=None, label: str | None = None,
               scale: float = 1.0):
    """The attention-output rule (see module docstring); returns the max-relative error against ``ref``.
    On the last R dims (rotated back by the inverse RoPE after a first rounding) the allowance also holds
    two ulps of the rotated pair's norm: a one-ulp flip of the partner element before the rotation enters
    this element through the rotation.  ``exact``: the oracle's un-rounded output (exact_output), checked on
    the first D - R dims within TOL * max|exact row| + half an ulp.  ``label`` records the errors in WORST.
    ``scale`` multiplies the allowance: 2 compares two GPU results that are each held to the rule against the
    same oracle (|a - b| <= |a - o| + |o - b|)."""
    g, r = f64(gpu), f64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    rowmax = np.abs(r).max(axis=-1, keepdims=True)
    allow = np.maximum(TOL[dtype] * rowmax, ulp(r, dtype))
    if R:
        D = r.shape[-1]
        pn = np.sqrt(r[..., D - R::2] ** 2 + r[..., D - R + 1::2] ** 2)
        allow[..., D - R:] += 2 * ulp(np.repeat(pn, 2, axis=-1), dtype)
    allow = allow * scale
    bad = np.abs(g - r) > allow
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at {tuple(idx)}: "
                             f"gpu {g[tuple(idx)]} oracle {r[tuple(idx)]} allow {allow[tuple(idx)]}")
    den = np.where(rowmax == 0, 1.0, rowmax)
    worst = float((np.abs(g - r) / den).max()) if g.size else 0.0
    rows = int(np.prod(g.shape[:-1])) if g.ndim > 1 else 1
    if exact is not None:
        e = f64(exact)
        assert e.shape == g.shape, (e.shape, g.shape)
        nd = e.shape[-1] - R
        emax = np.abs(e).max(axis=-1, keepdims=True)
        ge, ee = g[..., :nd], e[..., :nd]
        allow_e = TOL[dtype] * emax + 0.5 * ulp(ee, dtype)
        bad = np.abs(ge - ee) > allow_e
        if bad.any():
            idx = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: {bad.sum()} non-rope elements beyond TOL + half an ulp of the un-rounded "
                                 f"oracle; first at {tuple(idx)}: gpu {ge[tuple(idx)]} exact {ee[tuple(idx)]} "
                                 f"allow {allow_e[tuple(idx)]}")
        eden = np.where(emax == 0, 1.0, emax)
        if label and ge.size:
            _record(label, "exact_nonrope", float((np.abs(ge - ee) / eden).max()), 0)
            beyond = np.maximum(np.abs(ge - ee) - 0.5 * ulp(ee, dtype), 0.0)
            _record(label, "beyond_rounding", float((beyond / eden).max()), 0)
    if label:
        _record(label, "rounded", worst, rows)
    return worst


def check_pool_rows(gpu, ref, dtype: str, what: str = "pool", R: int = 0):
    """Rows both sides pooled from the SAME projections (bf16): per element within 2 ulps of the model
    dtype (the pooled value and the norm output are each rounded once, and may flip by one ulp between fp32
    and float64 arithmetic), plus, on the last R (rotated) dims, 2 ulps of the larger element of the rotated
    pair (a flip of the partner enters through the rotation), plus 2^-20 of the row's largest element for
    values a rotation cancels to near zero.  fp32 storage: 1e-5 of the row's largest element."""
    g, r = f64(gpu), f64(ref)
    rowmax = np.abs(r).max(axis=-1, keepdims=True)
    if dtype == "bf16":
        allow = 2 * ulp(r, dtype) + 2.0 ** -20 * rowmax
        if R:
            D = r.shape[-1]
            a, b = np.abs(r[..., D - R::2]), np.abs(r[..., D - R + 1::2])
            pm = np.repeat(np.maximum(a, b), 2, axis=-1)
            allow[..., D - R:] += 2 * ulp(pm, dtype)
        bad = np.abs(g - r) > allow
    else:
        bad = np.abs(g - r) > 1e-5 * rowmax + 1e-30
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements differ; first at {tuple(idx)}: gpu {g[tuple(idx)]} "
                             f"oracle {r[tuple(idx)]}")


def check_projection(gpu, ref, abs_dot, dtype: str, what: str = "projection"):
    """kv | gate projections: the GPU accumulates in fp32, the oracle in float64, and both round once to the
    model dtype.  They may land one ulp apart, or differ by the fp32 accumulation error, bounded here by
    2^-16 of sum_k |w_k x_k| (``abs_dot``); for fp32 storage, 1e-5 of that sum."""
    g, r = f64(gpu), f64(ref)
    if dtype == "bf16":
        allow = ulp(r, dtype) + 2.0 ** -16 * abs_dot
    else:
        allow = 1e-5 * abs_dot
    bad = np.abs(g - r) > allow
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements differ by more than one rounding; first at "
                             f"{tuple(idx)}: gpu {g[tuple(idx)]} oracle {r[tuple(idx)]}")


def oracle_compress_checked(layer, comp, x, pos, frontier, pool, n_rows, invf, gpu_proj, what):
    """Check the GPU's projections of x against the oracle's, then let the oracle pool the GPU's
    projections (so a one-ulp rounding flip upstream cannot masquerade as a pooling error)."""
    kv_o, g_o = O.project(layer, comp, x)
    ax = np.abs(np.asarray(x, dtype=np.float64))
    abs_dot = np.concatenate([ax @ np.abs(comp.wkv).T, ax @ np.abs(comp.wgate).T], axis=-1)
    gp = f64(gpu_proj)
    check_projection(gp, np.concatenate([kv_o, g_o], axis=-1), abs_dot, layer.dtype, what=f"{what} projection")
    Ld = kv_o.shape[-1]
    return O.compress_append(layer, comp, x, pos, frontier, pool, n_rows, invf, proj=(gp[..., :Ld], gp[..., Ld:]))


def pool_from_x_allowance(layer, comp, x, invf):
    """Bound on |GPU row - oracle row| when each side pools its OWN projections of the same hidden states x
    [1, T, X] (tokens 0 .. T-1 of one sequence from an empty cache), derived by propagating the projection
    rule through each step of the row's definition.  Returns (oracle rows [n, d], allowance [n, d]).

    With a_e, b_e the projection allowances of an entry's kv and gate (one ulp plus the fp32 accumulation term
    of check_projection), the softmax weights w_e over the window's entries and the pooled u = sum w_e kv_e:
      * kv:   sum_e w_e a_e
      * gate: dw_e = w_e (ds_e - sum_f w_f ds_f), and sum_e dw_e = 0, so |du| <= sum_e w_e |kv_e - u| (b_e + max_f b_f)
      * the GPU's fp32 pooling: 2^-20 sum_e w_e |kv_e| (fp32 carries 24 bits)
      * rounding u on either side: one ulp of the model dtype at |u| + du (|rnd(a) - rnd(b)| <= |a - b| + ulp)
      * RMSNorm y = u w / r, r = sqrt(mean u^2 + eps): |dy_c| <= |w_c| U_c / r + |y_c| rms(U) / r, then one ulp
      * RoPE at j * ratio rotates each pair: |d rot| <= |(dY_a, dY_b)| plus 2^-20 of the pair for the angle's
        fp32 sin/cos, then one ulp; other dims pass through (already in the model dtype)
    The first-order terms are scaled by 1.25 to cover second-order products."""
    dt = layer.dtype
    bits_rel = 2.0 ** -16 if dt == "bf16" else 1e-5
    x = np.asarray(x, dtype=np.float64)[0]
    T = x.shape[0]
    kv, g = O.project(layer, comp, x[None])
    kv, g = kv[0], g[0]
    ax = np.abs(x)
    a_kv = (ulp(kv, dt) if dt == "bf16" else 0.0) + bits_rel * (ax @ np.abs(comp.wkv).T)
    a_g = (ulp(g, dt) if dt == "bf16" else 0.0) + bits_rel * (ax @ np.abs(comp.wgate).T)
    tok = {t: (kv[t], g[t]) for t in range(T)}
    atok = {t: (a_kv[t], a_g[t]) for t in range(T)}
    no_ape = O.Compressor(wkv=comp.wkv, wgate=comp.wgate, ape=np.zeros_like(comp.ape), norm_w=comp.norm_w,
                          d=comp.d)
    n = T // layer.ratio
    d, R = comp.d, layer.R
    rows = np.zeros((n, d))
    allow = np.zeros((n, d))
    wn = np.asarray(comp.norm_w, dtype=np.float64)
    for j in range(n):
        kvj, sj = O.window_entries(layer, comp, j, tok)
        akv, ag = O.window_entries(layer, no_ape, j, atok)
        w = O.pool_weights(sj)
        u = (w * kvj).sum(axis=0)
        du = (w * akv).sum(axis=0) + (w * np.abs(kvj - u) * (ag + ag.max(axis=0))).sum(axis=0)
        du = 1.25 * du + 2.0 ** -20 * (w * np.abs(kvj)).sum(axis=0)
        U = du + ulp(np.abs(u) + du, dt)
        ur = O.store(u, dt)
        r = np.sqrt(np.mean(ur * ur) + layer.rms_eps)
        y = ur * wn / r
        dy = 1.25 * (np.abs(wn) * U / r + np.abs(y) * np.sqrt(np.mean(U * U)) / r) + 2.0 ** -20 * np.abs(y)
        Y = dy + ulp(np.abs(y) + dy, dt)
        rows[j] = O.finalize_row(layer, comp, u, j, invf)
        Z = Y.copy()
        ya, yb = y[d - R::2], y[d - R + 1::2]
        pair = np.sqrt(Y[d - R::2] ** 2 + Y[d - R + 1::2] ** 2) + 2.0 ** -20 * np.sqrt(ya ** 2 + yb ** 2)
        Z[d - R::2] = pair + ulp(np.abs(rows[j, d - R::2]) + pair, dt)
        Z[d - R + 1::2] = pair + ulp(np.abs(rows[j, d - R + 1::2]) + pair, dt)
        allow[j] = Z
    return rows, allow


def check_pool_from_x(gpu_rows, oracle_rows, allow, what: str = "pool from x"):
    """GPU rows against the oracle's rows built from x alone, within pool_from_x_allowance; returns the largest
    |difference| / allowance (<= 1) and the share of elements that differ at all."""
    g = f64(gpu_rows)
    diff = np.abs(g - oracle_rows)
    bad = diff > allow
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements beyond the derived bound; first at {tuple(idx)}: gpu "
                             f"{g[tuple(idx)]} oracle {oracle_rows[tuple(idx)]} allow {allow[tuple(idx)]}")
    return float((diff / allow).max()), float((diff > 0).mean())


def check_topk(gpu_sel, scores, k: int, n_vis: int, what: str = "top-k"):
    """The gap rule; ``scores`` are the oracle's scores of rows 0 .. n_vis-1."""
    gsel = sorted(int(j) for j in gpu_sel if j >= 0)
    if n_vis <= k:
        assert gsel == list(range(n_vis)), f"{what}: dense regime must select all {n_vis} rows"
        return
    assert len(gsel) == k, f"{what}: {len(gsel)} rows selected, want {k}"
    assert len(set(gsel)) == k and all(0 <= j < n_vis for j in gsel), f"{what}: invalid rows"
    oracle_sel = list(O.topk_select(scores, k))
    order = np.lexsort((np.arange(n_vis), -scores))
    sk, sk1 = scores[order[k - 1]], scores[order[k]]
    if (sk - sk1) > 1e-3 * abs(sk):
        assert gsel == oracle_sel, f"{what}: set differs with a clear gap ({sk} vs {sk1})"
    else:
        hi = scores > sk + 1e-3 * abs(sk)
        lo = scores < sk - 1e-3 * abs(sk)
        s = set(gsel)
        assert all(j in s for j in np.nonzero(hi)[0]), f"{what}: a clearly-above row is missing"
        assert not any(j in s for j in np.nonzero(lo)[0]), f"{what}: a clearly-below row is selected"


def check_prefill_chunk(cfg, run, host, ch, out, sel, queries, label: str | None = None):
    """Oracle check of one prefill chunk at positions cfg.ctx .. cfg.ctx + T - 1 on a one-sequence cache (empty
    or synthetic; ratio 4 with the indexer, or any other ratio without it): the GPU's projections of the chunk,
    then, for each query in ``queries``, its selection (gap rule against the oracle's scores) and its output
    (against the oracle recomputed with the GPU's selection, rounded and un-rounded).
    Returns (oracle state after the chunk's compress calls, rows emitted, first new row, window ring after the
    chunk, worst max-relative output error)."""
    from tests._common import oracle_comp, oracle_layer, oracle_state
    layer = oracle_layer(cfg)
    ca = oracle_comp(run.ca_host)
    ci = oracle_comp(run.ci_host) if cfg.has_indexer else None
    invf = f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    sink = f64(csa_synth.sinks(cfg))
    st = {k: (None if v is None else v[0:1].copy()) for k, v in oracle_state(host).items()}
    x = f64(ch.x)
    pos0 = cfg.ctx
    n0 = st["n_rows"].copy()
    st["front_a"], st["pool"], n_a, e = oracle_compress_checked(layer, ca, x, st["pos"], st["front_a"], st["pool"],
                                                                n0, invf, run.projs["attn"].cpu(), "chunk attn")
    assert e == 0
    if ci is not None:
        st["front_i"], st["ikeys"], _, e = oracle_compress_checked(layer, ci, x, st["pos"], st["front_i"],
                                                                   st["ikeys"], n0, invf, run.projs["index"].cpu(),
                                                                   "chunk index")
        assert e == 0
    T = ch.q.shape[0]
    n = int(n_a[0])
    lo = pos0 // cfg.ratio
    q, kv = f64(ch.q), f64(ch.kv)
    iq, iw = (f64(ch.iq), f64(ch.iw)) if ci is not None else (None, None)
    window = st["window"][0]
    pool = st["pool"][0]
    ikeys = st["ikeys"][0] if ci is not None else None
    kvr = [O.store(O.rope(kv[i], pos0 + i, invf), layer.dtype) for i in range(T)]
    gsel = sel.cpu().numpy()
    gout = out.cpu()
    worst = 0.0
    for i in queries:
        p = pos0 + i
        nv = O.visible_rows(layer, n, p)
        if ci is not None:
            rows = gsel[i][gsel[i] >= 0]
            scores = O.index_scores(layer, iq[i], iw[i], ikeys[:nv], p, invf) if nv > layer.topk else None
            check_topk(rows, scores, layer.topk, nv, what=f"query {i} top-k")
            rows = np.sort(rows)
        else:
            rows = np.arange(nv)
        win = [window[t % cfg.W] if t < pos0 else kvr[t - pos0] for t in O.window_tokens(layer, p)]
        keys = np.concatenate([pool[rows], np.stack(win)])
        qr = O.store(O.rope(q[i], p, invf), layer.dtype)
        o = O.attend(layer, qr, keys, sink)
        worst = max(worst, check_rows(gout[i], O.output_rows(layer, o, p, invf), layer.dtype,
                                      what=f"query {i} output", R=cfg.R, exact=exact_output(o, p, invf), label=label))
    ring = np.array(window)
    for t in range(max(pos0, pos0 + T - cfg.W), pos0 + T):
        ring[t % cfg.W] = kvr[t - pos0]
    return st, n, lo, ring, worst


def rel_metric(gpu, ref):
    g, r = f64(gpu), f64(ref)
    den = np.abs(r).max(axis=-1)
    den = np.where(den == 0, 1.0, den)
    return float((np.abs(g - r).max(axis=-1) / den).max())


class Runner:
    """Holds the device weights of one config and runs decode steps / prefill chunks."""

    def __init__(self, cfg: csa_synth.Config):
        self.cfg = cfg
        self.L = lib_layer(cfg)
        self.ca_host = csa_synth.compressor(cfg, "attn")
        self.ci_host = csa_synth.compressor(cfg, "index") if cfg.has_indexer else None
        self.ca = lib_comp(self.ca_host)
        self.ci = lib_comp(self.ci_host) if cfg.has_indexer else None
        self.sink = dev(csa_synth.sinks(cfg))
        self.inv_freq = dev(csa_synth.inv_freq(cfg))
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def compress(self, st: DevCache, x):
        """Both compress calls; returns the GPU's projections of the new tokens per pool.  A single new token's
        projection is read from its frontier slot (slot pos mod F); a chunk's from the call's workspace
        (layout: [B] int32 flags, then 256-byte aligned [B*T, 2*L*d] projections)."""
        x = dev(x)
        B, T = x.shape[0], x.shape[1]
        n0 = st.n_rows.clone()
        projs = {}
        pools = [("attn", self.ca, st.front_attn, st.pool, st.n_rows)]
        if self.cfg.has_indexer:
            pools.append(("index", self.ci, st.front_index, st.ikeys, n0))
        es = 2 if self.cfg.dtype == "bf16" else 4
        for name, comp, front, pool, n in pools:
            ws = torch.zeros(csa.workspace_size(self.L, csa.OP_COMPRESS, B, T, pool.shape[1]), dtype=torch.uint8,
                             device="cuda")
            csa.compress_append(self.L, comp, x, st.pos, front, pool, n, self.inv_freq, ws=ws, err=self.err)
            width = 2 * self.cfg.lanes * comp.d
            if T == 1:
                slots = (st.pos.long() % front.shape[1])
                projs[name] = front[torch.arange(B, device=front.device), slots].view(B, 1, width).clone()
            else:
                off = (4 * B + 255) // 256 * 256
                raw = ws[off:off + B * T * width * es]
                projs[name] = raw.view(self.cfg.storage).view(B, T, width).clone()
        return projs

    def compress_pair(self, st: DevCache, x):
        """csa_compress_append_pair (both pools, one call); returns the GPU's projections of the new tokens per
        pool, read from their frontier slots (slot (pos + i) mod F; the block fits the frontier)."""
        x = dev(x)
        B, T = x.shape[0], x.shape[1]
        F = st.front_attn.shape[1]
        assert T <= F
        n_i = st.n_rows.clone()
        ws = torch.zeros(csa.workspace_size(self.L, csa.OP_COMPRESS_PAIR, B, T, st.pool.shape[1]), dtype=torch.uint8,
                         device="cuda")
        csa.compress_append_pair(self.L, self.ca, self.ci, x, st.pos, st.front_attn, st.pool, st.n_rows,
                                 st.front_index, st.ikeys, n_i, self.inv_freq, ws=ws, err=self.err)
        torch.cuda.synchronize()
        assert torch.equal(n_i, st.n_rows)
        slots = (st.pos.long()[:, None] + torch.arange(T, device="cuda")[None]) % F
        rows = torch.arange(B, device="cuda")[:, None]
        return {"attn": st.front_attn[rows, slots].clone(), "index": st.front_index[rows, slots].clone()}

    def compress_and_index_overlapped(self, st: DevCache, si: csa_synth.StepInputs, sel, n_sel):
        """The index pool's compress call on a second stream while csa_index_topk_overlapped scans on the main
        stream (after the attention pool's compress call), joined by an event; sets self.projs."""
        x = dev(si.x)
        B = x.shape[0]
        n_idx = st.n_rows.clone()
        main = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(main)
        ready = torch.cuda.Event()
        mk = lambda pool: torch.zeros(csa.workspace_size(self.L, csa.OP_COMPRESS, B, 1, pool.shape[1]),  # noqa: E731
                                      dtype=torch.uint8, device="cuda")
        ws_i, ws_a = mk(st.ikeys), mk(st.pool)
        with torch.cuda.stream(side):
            csa.compress_append(self.L, self.ci, x, st.pos, st.front_index, st.ikeys, n_idx, self.inv_freq, ws=ws_i,
                                err=self.err)
            ready.record(side)
        csa.compress_append(self.L, self.ca, x, st.pos, st.front_attn, st.pool, st.n_rows, self.inv_freq, ws=ws_a,
                            err=self.err)
        csa.index_topk_overlapped(self.L, dev(si.iq), dev(si.iw), st.ikeys, n_idx, st.pos, self.inv_freq, sel, n_sel,
                                  pool_ready=ready, err=self.err)
        main.wait_stream(side)
        slots = st.pos.long() % st.front_attn.shape[1]
        rows = torch.arange(B, device="cuda")
        self.projs = {"attn": st.front_attn[rows, slots].view(B, 1, -1).clone(),
                      "index": st.front_index[rows, slots].view(B, 1, -1).clone()}

    def compress_pair_and_index_one_stream(self, st: DevCache, si: csa_synth.StepInputs, sel, n_sel):
        """Both pools through csa_compress_append_pair, then csa_index_topk_overlapped on the same stream with no
        event: its scan of the rows complete before the token runs beside the compress call's kernels."""
        x = dev(si.x)
        B = x.shape[0]
        n_idx = st.n_rows.clone()
        csa.compress_append_pair(self.L, self.ca, self.ci, x, st.pos, st.front_attn, st.pool, st.n_rows,
                                 st.front_index, st.ikeys, n_idx, self.inv_freq, err=self.err)
        csa.index_topk_overlapped(self.L, dev(si.iq), dev(si.iw), st.ikeys, n_idx, st.pos, self.inv_freq, sel, n_sel,
                                  err=self.err)
        slots = st.pos.long() % st.front_attn.shape[1]
        rows = torch.arange(B, device="cuda")
        self.projs = {"attn": st.front_attn[rows, slots].view(B, 1, -1).clone(),
                      "index": st.front_index[rows, slots].view(B, 1, -1).clone()}

    def decode_step(self, st: DevCache, si: csa_synth.StepInputs, overlap=False):
        """One decode step.  overlap: False (compress calls, then csa_index_topk), True (the index pool's compress
        call on a second stream beside csa_index_topk_overlapped, joined by an event) or "one_stream" (the pair
        call, then csa_index_topk_overlapped on one stream)."""
        cfg = self.cfg
        B = si.q.shape[0]
        sel = n_sel = None
        if cfg.has_indexer:
            sel = torch.empty(B, cfg.topk, dtype=torch.int32, device="cuda")
            n_sel = torch.empty(B, dtype=torch.int32, device="cuda")
        if overlap == "one_stream" and cfg.has_indexer:
            self.compress_pair_and_index_one_stream(st, si, sel, n_sel)
        elif overlap and cfg.has_indexer:
            self.compress_and_index_overlapped(st, si, sel, n_sel)
        else:
            self.projs = self.compress(st, si.x)
            if cfg.has_indexer:
                csa.index_topk(self.L, dev(si.iq), dev(si.iw), st.ikeys, st.n_rows, st.pos, self.inv_freq, sel,
                               n_sel, err=self.err)
        out = torch.empty(B, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
        csa.attend_decode(self.L, dev(si.q), dev(si.kv), self.sink, st.window, st.pool, st.n_rows, sel, n_sel,
                          st.pos, self.inv_freq, out, err=self.err)
        st.pos += 1
        return out, sel, n_sel

    def prefill(self, st: DevCache, ch: csa_synth.StepInputs, pos0: int):
        cfg = self.cfg
        T = ch.q.shape[0]
        self.projs = self.compress(st, ch.x)
        out = torch.empty(T, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
        sel = torch.empty(T, max(cfg.topk, 1), dtype=torch.int32, device="cuda")
        csa.attend_prefill_chunk(self.L, dev(ch.q), dev(ch.kv), dev(ch.iq), dev(ch.iw), self.sink, pos0,
                                 st.window[0], st.pool[0], st.ikeys[0] if st.ikeys is not None else None,
                                 st.n_rows, self.inv_freq, out, sel_out=sel, err=self.err)
        st.pos += T
        return out, sel
