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
                     topk=cfg.topk, X=cfg.X, scale=cfg.scale, rms_eps=cfg.rms_eps)


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


def check_rows(gpu, ref, dtype: str, what: str = "output", R: int = 0):
    """The attention-output rule (see module docstring); returns the max-relative error.
    On the last R dims (rotated back by the inverse RoPE after a first rounding) the allowance also holds
    two ulps of the rotated pair's norm: a one-ulp flip of the partner element before the rotation enters
    this element through the rotation."""
    g, r = f64(gpu), f64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    rowmax = np.abs(r).max(axis=-1, keepdims=True)
    allow = np.maximum(TOL[dtype] * rowmax, ulp(r, dtype))
    if R:
        D = r.shape[-1]
        pn = np.sqrt(r[..., D - R::2] ** 2 + r[..., D - R + 1::2] ** 2)
        allow[..., D - R:] += 2 * ulp(np.repeat(pn, 2, axis=-1), dtype)
    bad = np.abs(g - r) > allow
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at {tuple(idx)}: "
                             f"gpu {g[tuple(idx)]} oracle {r[tuple(idx)]} allow {allow[tuple(idx)]}")
    den = np.where(rowmax == 0, 1.0, rowmax)
    return float((np.abs(g - r) / den).max()) if g.size else 0.0


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

    def decode_step(self, st: DevCache, si: csa_synth.StepInputs, overlap: bool = False):
        cfg = self.cfg
        B = si.q.shape[0]
        sel = n_sel = None
        if cfg.has_indexer:
            sel = torch.empty(B, cfg.topk, dtype=torch.int32, device="cuda")
            n_sel = torch.empty(B, dtype=torch.int32, device="cuda")
        if overlap and cfg.has_indexer:
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
