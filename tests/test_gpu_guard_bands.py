"""Guard bands around every buffer the library reads or writes: a stand-in for a memory checker (compute-sanitizer
is not available here).

Each buffer (inputs, pools, frontier and window rings, row counts, positions, selections, outputs, workspaces, the
error word) is a view into a larger allocation whose 4 KB margins before and after hold 0xFF bytes; after the calls
every margin must still hold them, so no kernel wrote outside its buffer, and every float the calls produced must be
finite: 0xFF bytes read as bf16 or fp32 are NaN, so a kernel reading a float input outside its buffer would carry a
NaN into its outputs.  The calls run on small, ragged
shapes that reach every kernel family: single-token and chunk compression (both pools, the pair call, fp8 index
rows), decode, prefill chunks, verify blocks, packed varlen batches, the trim, the fp8 conversion and a ratio-128
layer.
"""
import dataclasses

import pytest
import torch

import csa_synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests import _gpu as G

GUARD = 4096      # bytes on each side (a multiple of 256: the view keeps the allocation's alignment)
PATTERN = 0xFF    # NaN as bf16 / fp32, -1 as int32


class Guards:
    def __init__(self):
        self.slabs = []

    def wrap(self, name, t):
        """A device copy of t inside a guarded slab."""
        t = t.to("cuda").contiguous()
        nb = t.numel() * t.element_size()
        slab = torch.full((2 * GUARD + nb,), PATTERN, dtype=torch.uint8, device="cuda")
        view = slab[GUARD:GUARD + nb].view(t.dtype).view(t.shape)
        view.copy_(t)
        self.slabs.append((name, slab, nb, view))
        return view

    def empty(self, name, shape, dtype):
        return self.wrap(name, torch.zeros(shape, dtype=dtype))

    def ws(self, name, nbytes):
        return self.wrap(name, torch.zeros(max(int(nbytes), 256), dtype=torch.uint8))

    def inp(self, t, name="input"):
        """An input, guarded."""
        return self.wrap(f"{name}{len(self.slabs)}", t)

    def weights(self, run):
        """The runner's compressor weights, sinks and inverse frequencies, guarded."""
        def comp(c, tag):
            if c is None:
                return None
            return dataclasses.replace(c, wkv=self.wrap(tag + "wkv", c.wkv), wgate=self.wrap(tag + "wgate", c.wgate),
                                       ape=self.wrap(tag + "ape", c.ape), norm_w=self.wrap(tag + "norm_w", c.norm_w))
        run.ca, run.ci = comp(run.ca, "ca_"), comp(run.ci, "ci_")
        run.sink, run.inv_freq = self.wrap("sink", run.sink), self.wrap("inv_freq", run.inv_freq)
        return run

    def finite(self, *fp8_rows):
        """Every guarded float buffer (inputs, weights, caches, outputs) holds finite values only; so do the scales
        (fp32 at byte 128) of the named fp8 index-row buffers."""
        torch.cuda.synchronize()
        for name, _, _, t in self.slabs:
            if t.dtype.is_floating_point:
                bad = (~torch.isfinite(t.float())).sum().item()
                assert bad == 0, f"{name}: {bad} values not finite"
        for name, t in fp8_rows:
            bad = (~torch.isfinite(t[..., 128:132].contiguous().view(torch.float32))).sum().item()
            assert bad == 0, f"{name}: {bad} scales not finite"

    def check(self):
        torch.cuda.synchronize()
        for name, slab, nb, _ in self.slabs:
            head, tail = slab[:GUARD], slab[GUARD + nb:]
            for part, where in ((head, "before"), (tail, "after")):
                bad = torch.nonzero(part != PATTERN)
                assert bad.numel() == 0, (f"{name}: {bad.numel()} bytes changed {where} the buffer (first at offset "
                                          f"{int(bad[0])})")


def _cache(gd, cfg, host, pre=""):
    """The written state of a cache, guarded."""
    st = G.DevCache(host)
    for k in ("pool", "ikeys", "window", "front_attn", "front_index", "n_rows", "pos"):
        v = getattr(st, k)
        if v is not None:
            setattr(st, k, gd.wrap(pre + k, v))
    return st


def test_guard_bands_decode_pair_verify_and_trim():
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=3, ctx=2045, rollback=8)
    cap = cfg.ctx // 4 + 40
    run = G.Runner(cfg)
    gd = Guards()
    gd.weights(run)
    st = _cache(gd, cfg, csa_synth.synth_cache(cfg, cap))
    err = gd.empty("err", (1,), torch.int32)
    B = cfg.B
    for k in range(6):  # decode steps across window completions and the dense -> sparse threshold
        si = csa_synth.step_inputs(cfg.replace(cid=cfg.cid + 700), k)
        n_i = st.n_rows.clone()
        ws_p = gd.ws(f"ws_pair{k}", csa.workspace_size(run.L, csa.OP_COMPRESS_PAIR, B, 1, cap))
        csa.compress_append_pair(run.L, run.ca, run.ci, gd.inp(si.x), st.pos, st.front_attn, st.pool, st.n_rows,
                                 st.front_index, st.ikeys, n_i, run.inv_freq, ws=ws_p, err=err)
        sel = gd.empty(f"sel{k}", (B, cfg.topk), torch.int32)
        n_sel = gd.empty(f"n_sel{k}", (B,), torch.int32)
        ws_i = gd.ws(f"ws_index{k}", csa.workspace_size(run.L, csa.OP_INDEX_TOPK, B, 1, cap))
        csa.index_topk(run.L, gd.inp(si.iq), gd.inp(si.iw), st.ikeys, st.n_rows, st.pos, run.inv_freq, sel, n_sel,
                       ws=ws_i, err=err)
        sel_s = gd.empty(f"sel_static{k}", (B, cfg.topk), torch.int32)
        n_sel_s = gd.empty(f"n_sel_static{k}", (B,), torch.int32)
        csa.index_topk_static(run.L, gd.inp(si.iq), gd.inp(si.iw), st.ikeys, st.n_rows, st.pos, run.inv_freq, sel_s,
                              n_sel_s, err=err)
        out = gd.empty(f"out{k}", (B, cfg.H, cfg.D), cfg.storage)
        ws_a = gd.ws(f"ws_attend{k}", csa.workspace_size(run.L, csa.OP_ATTEND_DECODE, B, 1, cap))
        csa.attend_decode(run.L, gd.inp(si.q), gd.inp(si.kv), run.sink, st.window, st.pool, st.n_rows, sel, n_sel,
                          st.pos, run.inv_freq, out, ws=ws_a, err=err)
        csa.advance_positions(st.pos, 1)
    # a verify block of T = 4 tokens, then a trim of the last two
    T = 4
    blk = [csa_synth.step_inputs(cfg.replace(cid=cfg.cid + 710), i) for i in range(T)]
    x = torch.cat([b.x for b in blk], dim=1)
    n_i = st.n_rows.clone()
    ws_p = gd.ws("ws_pair_block", csa.workspace_size(run.L, csa.OP_COMPRESS_PAIR, B, T, cap))
    csa.compress_append_pair(run.L, run.ca, run.ci, gd.inp(x), st.pos, st.front_attn, st.pool, st.n_rows,
                             st.front_index, st.ikeys, n_i, run.inv_freq, ws=ws_p, err=err)
    sel = gd.empty("sel_verify", (B, T, cfg.topk), torch.int32)
    n_sel = gd.empty("n_sel_verify", (B, T), torch.int32)
    ws_v = gd.ws("ws_verify_index", csa.workspace_size(run.L, csa.OP_INDEX_TOPK, B * T, 1, cap))
    csa.index_topk_verify(run.L, gd.inp(torch.stack([b.iq for b in blk], 1)),
                          gd.inp(torch.stack([b.iw for b in blk], 1)), st.ikeys, st.n_rows, st.pos, run.inv_freq, sel,
                          n_sel, ws=ws_v, err=err)
    out = gd.empty("out_verify", (B, T, cfg.H, cfg.D), cfg.storage)
    ws_va = gd.ws("ws_verify_attend", csa.workspace_size(run.L, csa.OP_ATTEND_DECODE, B * T, 1, cap))
    csa.attend_verify(run.L, gd.inp(torch.stack([b.q for b in blk], 1)), gd.inp(torch.stack([b.kv for b in blk], 1)),
                      run.sink, st.window, st.pool, st.n_rows, sel, n_sel, st.pos, run.inv_freq, out, ws=ws_va, err=err)
    csa.advance_positions(st.pos, T)
    hw = gd.wrap("hw", st.pos.clone())
    n_back = gd.wrap("n_back", torch.tensor([2, 0, 1], dtype=torch.int32))
    n_i = gd.wrap("n_rows_i_trim", st.n_rows.clone())
    csa.trim(run.L, n_back, st.pos, st.n_rows, n_i, hw, err=err)
    gd.check()
    gd.finite()
    assert err.item() == 0


def test_guard_bands_chunks_prefill_and_varlen():
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=1, ctx=1900)
    T = 301
    cap = (cfg.ctx + T) // 4 + 20
    run = G.Runner(cfg)
    gd = Guards()
    gd.weights(run)
    host = csa_synth.synth_cache(cfg, cap)
    st = _cache(gd, cfg, host)
    err = gd.empty("err", (1,), torch.int32)
    ch = csa_synth.chunk_inputs(cfg.replace(cid=cfg.cid + 720), T)
    n_i = st.n_rows.clone()
    for name, comp, front, pool, n in (("attn", run.ca, st.front_attn, st.pool, st.n_rows),
                                       ("index", run.ci, st.front_index, st.ikeys, n_i)):
        ws = gd.ws(f"ws_chunk_{name}", csa.workspace_size(run.L, csa.OP_COMPRESS, 1, T, cap))
        csa.compress_append(run.L, comp, gd.inp(ch.x), st.pos, front, pool, n, run.inv_freq, ws=ws, err=err)
    out = gd.empty("out_prefill", (T, cfg.H, cfg.D), cfg.storage)
    sel = gd.empty("sel_prefill", (T, cfg.topk), torch.int32)
    ws = gd.ws("ws_prefill", csa.workspace_size(run.L, csa.OP_ATTEND_PREFILL, 1, T, cap))
    csa.attend_prefill_chunk(run.L, gd.inp(ch.q), gd.inp(ch.kv), gd.inp(ch.iq), gd.inp(ch.iw), run.sink, cfg.ctx,
                             st.window[0], st.pool[0], st.ikeys[0], st.n_rows, run.inv_freq, out, sel_out=sel, ws=ws,
                             err=err)
    gd.check()
    gd.finite()
    assert err.item() == 0
    # a packed batch: a fresh prompt, an empty chunk, one token and a long chunk across dense -> sparse
    cfgv = csa_synth.CONFIGS[3].replace(B=4, ctx=0)
    lens, ctxs = [37, 0, 1, 260], [0, 400, 803, 1950]
    capv = (max(ctxs) + max(lens)) // 4 + 20
    runv = G.Runner(cfgv)
    hostv = csa_synth.empty_cache(cfgv, capv)
    for b, c in enumerate(ctxs):  # sequence b holds c tokens of synthetic rows
        hb = csa_synth.synth_cache(cfgv.replace(B=1, ctx=c), capv) if c else csa_synth.empty_cache(cfgv, capv, B=1)
        for k in ("pool", "ikeys", "window", "front_attn", "front_index", "n_rows", "pos"):
            getattr(hostv, k)[b] = getattr(hb, k)[0]
    gv = Guards()
    gv.weights(runv)
    sv = _cache(gv, cfgv, hostv)
    errv = gv.empty("err", (1,), torch.int32)
    N = sum(lens)
    cu = gv.wrap("cu_seqlens", torch.tensor([0] + list(torch.tensor(lens).cumsum(0)), dtype=torch.int32))
    chv = csa_synth.chunk_inputs(cfgv.replace(cid=cfgv.cid + 730), N)
    n_i = sv.n_rows.clone()
    for name, comp, front, pool, n in (("attn", runv.ca, sv.front_attn, sv.pool, sv.n_rows),
                                       ("index", runv.ci, sv.front_index, sv.ikeys, n_i)):
        ws = gv.ws(f"ws_varlen_{name}", csa.workspace_size(runv.L, csa.OP_COMPRESS_VARLEN, 4, N, capv))
        csa.compress_append_varlen(runv.L, comp, gv.inp(chv.x[0]), cu, max(lens), sv.pos, front, pool, n,
                                   runv.inv_freq, ws=ws, err=errv)
    out = gv.empty("out_varlen", (N, cfgv.H, cfgv.D), cfgv.storage)
    sel = gv.empty("sel_varlen", (N, cfgv.topk), torch.int32)
    ws = gv.ws("ws_varlen_attend", csa.workspace_size(runv.L, csa.OP_ATTEND_PREFILL_VARLEN, 4, N, capv))
    csa.attend_prefill_varlen(runv.L, gv.inp(chv.q), gv.inp(chv.kv), gv.inp(chv.iq), gv.inp(chv.iw), runv.sink, cu,
                              max(lens), sv.pos, sv.window, sv.pool, sv.ikeys, sv.n_rows, runv.inv_freq, out,
                              sel_out=sel, ws=ws, err=errv)
    gv.check()
    gv.finite()
    assert errv.item() == 0


def test_guard_bands_fp8_rows_and_ratio128():
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=2, ctx=0)
    T0 = 2051
    cap = (T0 + 8) // 4 + 30
    run = G.Runner(cfg)
    L8 = dataclasses.replace(run.L, index_fp8=True)
    gd = Guards()
    gd.weights(run)
    host = csa_synth.empty_cache(cfg, cap)
    st = _cache(gd, cfg, host)
    st.ikeys = gd.empty("ikeys_fp8", (cfg.B, cap, csa.FP8_ROW_BYTES), torch.uint8)
    err = gd.empty("err", (1,), torch.int32)
    x = csa_synth.hidden(cfg, T0, tag=41)
    n_i = st.n_rows.clone()
    for name, comp, front, pool, n in (("attn", run.ca, st.front_attn, st.pool, st.n_rows),
                                       ("index", run.ci, st.front_index, st.ikeys, n_i)):
        ws = gd.ws(f"ws_chunk_{name}", csa.workspace_size(L8, csa.OP_COMPRESS, cfg.B, T0, cap))
        csa.compress_append(L8, comp, gd.inp(x), st.pos, front, pool, n, run.inv_freq, ws=ws, err=err)
    st.pos += T0
    for k in range(5):
        si = csa_synth.step_inputs(cfg.replace(cid=cfg.cid + 740), k)
        n_i = st.n_rows.clone()
        ws_p = gd.ws(f"ws_pair{k}", csa.workspace_size(L8, csa.OP_COMPRESS_PAIR, cfg.B, 1, cap))
        csa.compress_append_pair(L8, run.ca, run.ci, gd.inp(si.x), st.pos, st.front_attn, st.pool, st.n_rows,
                                 st.front_index, st.ikeys, n_i, run.inv_freq, ws=ws_p, err=err)
        sel = gd.empty(f"sel{k}", (cfg.B, cfg.topk), torch.int32)
        n_sel = gd.empty(f"n_sel{k}", (cfg.B,), torch.int32)
        ws_i = gd.ws(f"ws_index{k}", csa.workspace_size(L8, csa.OP_INDEX_TOPK, cfg.B, 1, cap))
        csa.index_topk(L8, gd.inp(si.iq), gd.inp(si.iw), st.ikeys, st.n_rows, st.pos, run.inv_freq, sel, n_sel, ws=ws_i,
                       err=err)
        st.pos += 1
    src = gd.inp(csa_synth.synth_cache(cfg.replace(ctx=4 * 77), 77).ikeys)
    dst = gd.empty("rows_fp8", (cfg.B, 77, csa.FP8_ROW_BYTES), torch.uint8)
    csa.index_rows_fp8(L8, src, dst)
    gd.check()
    gd.finite(("ikeys_fp8", st.ikeys), ("rows_fp8", dst))
    assert err.item() == 0
    # a ratio-128 layer: chunk compression across a window boundary, decode attention over every row
    c4 = csa_synth.CONFIGS[4].replace(B=2, ctx=128 * 40 - 3)
    cap4 = c4.ctx // 128 + 8
    r4 = G.Runner(c4)
    g4 = Guards()
    g4.weights(r4)
    s4 = _cache(g4, c4, csa_synth.synth_cache(c4, cap4))
    err4 = g4.empty("err", (1,), torch.int32)
    for k in range(5):
        si = csa_synth.step_inputs(c4.replace(cid=c4.cid + 750), k)
        ws = g4.ws(f"ws_compress{k}", csa.workspace_size(r4.L, csa.OP_COMPRESS, c4.B, 1, cap4))
        csa.compress_append(r4.L, r4.ca, g4.inp(si.x), s4.pos, s4.front_attn, s4.pool, s4.n_rows, r4.inv_freq, ws=ws,
                            err=err4)
        out = g4.empty(f"out{k}", (c4.B, c4.H, c4.D), c4.storage)
        ws_a = g4.ws(f"ws_attend{k}", csa.workspace_size(r4.L, csa.OP_ATTEND_DECODE, c4.B, 1, cap4))
        csa.attend_decode(r4.L, g4.inp(si.q), g4.inp(si.kv), r4.sink, s4.window, s4.pool, s4.n_rows, None, None, s4.pos,
                          r4.inv_freq, out, ws=ws_a, err=err4)
        csa.advance_positions(s4.pos, 1)
    g4.check()
    g4.finite()
    assert err4.item() == 0
