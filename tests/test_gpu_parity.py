"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Inputs are the seeded synthetic workloads of csa_synth (configs 1-5 and small
variants); comparison rules are in tests/_gpu.py.
"""
import numpy as np
import pytest
import torch

import csa_synth
from oracle import csa_oracle as O
from tests._common import f64, oracle_comp, oracle_layer, oracle_state

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests import _gpu as G


def _oracle_seq_state(cache: csa_synth.Cache, b: int) -> dict:
    """Oracle state of sequence b alone (converted after slicing: a full config-3 cache in float64 is ~1.3 GB)."""
    one = csa_synth.Cache(**{k: (None if v is None else v[b:b + 1]) for k, v in vars(cache).items()})
    return oracle_state(one)


def _step_rows(si: csa_synth.StepInputs, b: int):
    return (f64(si.x[b:b + 1]), f64(si.q[b:b + 1]), f64(si.kv[b:b + 1]), f64(si.iq[b:b + 1]), f64(si.iw[b:b + 1]))


def _seq_projs(run, b):
    return {k: v[b:b + 1].cpu() for k, v in run.projs.items()}


def _exact_decode_output(layer, q, sink, window, pool, n_rows, sel, n_sel, p, invf):
    """The un-rounded oracle output of one decode query: the keys of O.attend_decode (selected rows, then the
    window tokens, the new token already in the ring), float64 attention, rotated back."""
    rows = np.arange(O.visible_rows(layer, int(n_rows), p)) if sel is None else \
        np.asarray(sel[:int(n_sel)], dtype=np.int64)
    keys = np.concatenate([pool[rows]] +
                          [window[t % layer.W][None] for t in O.window_tokens(layer, p)])
    o = O.attend(layer, O.store(O.rope(q, p, invf), layer.dtype), keys, sink)
    return G.exact_output(o, p, invf)


def _oracle_decode_check(layer, ca, ci, st, xs, sink, invf, gpu_out, gpu_sel, gpu_nsel, what, projs, label=None):
    """Advance the oracle state by one token and check the GPU's projections, selection and output for it
    (against the rounded and the un-rounded oracle output).  ``projs`` are the GPU's projections of this
    sequence's token (per pool); ``label`` records the errors under that workload name."""
    x, q, kv, iq, iw = xs
    n0 = st["n_rows"].copy()
    st["front_a"], st["pool"], n_a, e1 = G.oracle_compress_checked(layer, ca, x, st["pos"], st["front_a"],
                                                                   st["pool"], n0, invf, projs["attn"], what)
    assert e1 == 0
    sel = n_sel = None
    if layer.has_indexer:
        st["front_i"], st["ikeys"], n_i, e2 = G.oracle_compress_checked(layer, ci, x, st["pos"], st["front_i"],
                                                                        st["ikeys"], n0, invf, projs["index"], what)
        assert e2 == 0 and np.array_equal(n_a, n_i)
        p = int(st["pos"][0])
        nv = O.visible_rows(layer, int(n_a[0]), p)
        scores = O.index_scores(layer, iq[0], iw[0], st["ikeys"][0, :nv], p, invf) if nv > layer.topk else None
        G.check_topk(gpu_sel[:int(gpu_nsel)], scores, layer.topk, nv, what=f"{what} top-k")
        sel = np.asarray(gpu_sel, dtype=np.int64)[None]
        n_sel = np.array([int(gpu_nsel)])
    st["n_rows"] = n_a
    out, st["window"], err = O.attend_decode(layer, q, kv, sink, st["window"], st["pool"], n_a, sel, n_sel, st["pos"],
                                             invf)
    assert err == 0
    p = int(st["pos"][0])
    exact = _exact_decode_output(layer, q[0], sink, st["window"][0], st["pool"][0], n_a[0],
                                 None if sel is None else sel[0], None if n_sel is None else n_sel[0], p, invf)
    st["pos"] = st["pos"] + 1
    return G.check_rows(gpu_out, out[0], layer.dtype, what=f"{what} output", R=layer.R, exact=exact, label=label)


def test_config1_tiny_fp32_decode_256_steps():
    """Config 1: fp32 storage, 256 decode steps from an empty cache (sparse from step 68), every step checked."""
    cfg = csa_synth.CONFIGS[1]
    cap = cfg.steps // cfg.ratio + 2
    run = G.Runner(cfg)
    host = csa_synth.empty_cache(cfg, cap)
    st_g = G.DevCache(host)
    layer = oracle_layer(cfg)
    ca, ci = oracle_comp(run.ca_host), oracle_comp(run.ci_host)
    sink, invf = f64(csa_synth.sinks(cfg)), f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    st_o = _oracle_seq_state(host, 0)
    worst = 0.0
    for step in range(cfg.steps):
        si = csa_synth.step_inputs(cfg, step)
        out, sel, n_sel = run.decode_step(st_g, si)
        torch.cuda.synchronize()
        worst = max(worst, _oracle_decode_check(layer, ca, ci, st_o, _step_rows(si, 0), sink, invf, out[0].cpu(),
                                                sel[0].cpu().numpy(), n_sel[0].item(), f"step {step}",
                                                _seq_projs(run, 0), label="1 tiny-f32-decode-256"))
    assert run.err.item() == 0
    n = int(st_o["n_rows"][0])
    assert n == cfg.steps // cfg.ratio == st_g.n_rows.item()
    G.check_pool_rows(st_g.pool[0, :n].cpu(), st_o["pool"][0, :n], "f32", "attention pool", R=cfg.R)
    G.check_pool_rows(st_g.ikeys[0, :n].cpu(), st_o["ikeys"][0, :n], "f32", "index pool", R=cfg.R)
    G.check_pool_rows(st_g.window[0].cpu(), st_o["window"][0], "f32", "window")
    # end to end from x: the oracle pools its own projections of the 256 tokens
    xs = np.concatenate([f64(csa_synth.step_inputs(cfg, step).x) for step in range(cfg.steps)], axis=1)
    for name, comp, got in (("attention pool", ca, st_g.pool), ("index pool", ci, st_g.ikeys)):
        rows, allow = G.pool_from_x_allowance(layer, comp, xs, invf)
        ratio, share = G.check_pool_from_x(got[0, :n].cpu(), rows, allow, what=f"{name} from x")
        print(f"config 1 {name} from x: largest |diff| / bound {ratio:.3f}, {100 * share:.1f} % of elements differ")
    print(f"config 1: worst max-relative output error {worst:.2e}")


def test_config2_flash_build_8k_then_decode():
    """Config 2: compress 8192 seeded hidden tokens into both pools, then one decode step at p = 8192."""
    cfg = csa_synth.CONFIGS[2]
    cap = cfg.prefill_tokens // cfg.ratio + 8
    run = G.Runner(cfg)
    host = csa_synth.empty_cache(cfg, cap)
    st_g = G.DevCache(host)
    xs = csa_synth.hidden(cfg, cfg.prefill_tokens)
    projs = run.compress(st_g, xs)
    st_g.pos += cfg.prefill_tokens
    layer = oracle_layer(cfg)
    ca, ci = oracle_comp(run.ca_host), oracle_comp(run.ci_host)
    st_o = _oracle_seq_state(host, 0)
    invf = f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    x = f64(xs)
    n0 = st_o["n_rows"].copy()
    st_o["front_a"], st_o["pool"], n_a, e = G.oracle_compress_checked(
        layer, ca, x, st_o["pos"], st_o["front_a"], st_o["pool"], n0, invf, projs["attn"].cpu(), "8k build attn")
    st_o["front_i"], st_o["ikeys"], n_i, _ = G.oracle_compress_checked(
        layer, ci, x, st_o["pos"], st_o["front_i"], st_o["ikeys"], n0, invf, projs["index"].cpu(), "8k build index")
    st_o["n_rows"], st_o["pos"] = n_a, st_o["pos"] + cfg.prefill_tokens
    torch.cuda.synchronize()
    assert e == 0 and int(n_a[0]) == 2048 == st_g.n_rows.item()
    G.check_pool_rows(st_g.pool[0, :2048].cpu(), st_o["pool"][0, :2048], "bf16", "attention pool", R=cfg.R)
    G.check_pool_rows(st_g.ikeys[0, :2048].cpu(), st_o["ikeys"][0, :2048], "bf16", "index pool", R=cfg.R)
    G.check_pool_rows(st_g.front_attn.cpu(), st_o["front_a"], "bf16", "attention frontier")
    # end to end from x: the oracle pools its own projections of the 8192 tokens (derived bound)
    for name, comp, got in (("attention pool", ca, st_g.pool), ("index pool", ci, st_g.ikeys)):
        rows, allow = G.pool_from_x_allowance(layer, comp, x, invf)
        ratio, share = G.check_pool_from_x(got[0, :2048].cpu(), rows, allow, what=f"{name} from x")
        print(f"config 2 {name} from x: largest |diff| / bound {ratio:.3f}, {100 * share:.1f} % of elements differ")
    # one decode step; window ring starts empty except what decode appends
    si = csa_synth.step_inputs(cfg, 0)
    out, sel, n_sel = run.decode_step(st_g, si)
    torch.cuda.synchronize()
    sink = f64(csa_synth.sinks(cfg))
    # the oracle continues from ITS pools (within 2 ulps of the GPU's)
    _oracle_decode_check(layer, ca, ci, st_o, _step_rows(si, 0), sink, invf, out[0].cpu(), sel[0].cpu().numpy(),
                         n_sel[0].item(), "config 2", _seq_projs(run, 0), label="2 flash-decode-b1-ctx8k")
    assert run.err.item() == 0


@pytest.mark.parametrize("cid,ctx,steps,seqs,overlap", [(3, 32768, 10, (0, 13, 31), False),
                                                         (3, 32768 + 1, 6, (5, 30), True),
                                                         (3, 32768 + 2, 6, (2, 19, 31), "one_stream"),
                                                         (4, 262144 - 3, 6, (0, 15), False)])
def test_batched_decode_sampled_sequences(cid, ctx, steps, seqs, overlap):
    """Configs 3 and 4 at full batch and context: every sequence runs on the GPU; the oracle follows
    a few of them step by step (window-boundary crossings included).  The second case drives the indexer
    through csa_index_topk_overlapped beside the index pool's compress call on another stream; the third
    through csa_compress_append_pair and csa_index_topk_overlapped on one stream (the bench's order)."""
    cfg = csa_synth.CONFIGS[cid]
    cap = ctx // cfg.ratio + steps // cfg.ratio + 4
    run = G.Runner(cfg)
    host = csa_synth.synth_cache(cfg, cap, ctx=ctx)
    st_g = G.DevCache(host)
    layer = oracle_layer(cfg)
    ca = oracle_comp(run.ca_host)
    ci = oracle_comp(run.ci_host) if cfg.has_indexer else None
    sink, invf = f64(csa_synth.sinks(cfg)), f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    st_o = {b: _oracle_seq_state(host, b) for b in seqs}
    for step in range(steps):
        si = csa_synth.step_inputs(cfg, step)
        out, sel, n_sel = run.decode_step(st_g, si, overlap=overlap)
        torch.cuda.synchronize()
        for b in seqs:
            _oracle_decode_check(layer, ca, ci, st_o[b], _step_rows(si, b), sink, invf, out[b].cpu(),
                                 None if sel is None else sel[b].cpu().numpy(),
                                 None if n_sel is None else n_sel[b].item(), f"cfg {cid} seq {b} step {step}",
                                 _seq_projs(run, b), label=f"{cid} {cfg.name}")
    assert run.err.item() == 0
    for b in seqs:
        n = int(st_o[b]["n_rows"][0])
        assert n == st_g.n_rows[b].item()
        lo = ctx // cfg.ratio
        G.check_pool_rows(st_g.pool[b, lo:n].cpu(), st_o[b]["pool"][0, lo:n], "bf16", "new pool rows", R=cfg.R)
        G.check_pool_rows(st_g.window[b].cpu(), st_o[b]["window"][0], "bf16", "window")


def _check_prefill(cfg, run, host, ch, out, sel, queries, label=None):
    return G.check_prefill_chunk(cfg, run, host, ch, out, sel, queries, label=label)


def test_config5_prefill_chunk_sampled_queries():
    """Config 5: a 4096-token chunk on a 65536-token cache.  All emitted rows, the frontier and the window
    are checked; the per-query selection and output are checked on sampled queries."""
    cfg = csa_synth.CONFIGS[5]
    cap = (cfg.ctx + cfg.T) // cfg.ratio + 4
    run = G.Runner(cfg)
    host = csa_synth.synth_cache(cfg, cap)
    st_g = G.DevCache(host)
    ch = csa_synth.chunk_inputs(cfg)
    out, sel = run.prefill(st_g, ch, cfg.ctx)
    torch.cuda.synchronize()
    assert run.err.item() == 0
    rng = np.random.default_rng(0)
    queries = sorted(set([0, 1, 2, 3, 4, 126, 127, 128, 129, 151, 152, 153, 303, 304, 2047, 4094, 4095] +
                         list(rng.integers(0, cfg.T, 12))))
    st, n, lo, ring, _ = _check_prefill(cfg, run, host, ch, out, sel, queries, label="5 flash-prefill-t4096-ctx64k")
    assert n == st_g.n_rows.item() == (cfg.ctx + cfg.T) // 4
    G.check_pool_rows(st_g.pool[0, lo:n].cpu(), st["pool"][0, lo:n], "bf16", "chunk pool rows", R=cfg.R)
    G.check_pool_rows(st_g.ikeys[0, lo:n].cpu(), st["ikeys"][0, lo:n], "bf16", "chunk index rows", R=cfg.R)
    G.check_pool_rows(st_g.front_index.cpu(), st["front_i"], "bf16", "index frontier")
    G.check_pool_rows(st_g.window[0].cpu(), ring, "bf16", "window after chunk")


def test_prefill_every_query_with_late_dominant_rows():
    """Every query of a 300-token chunk (two or more queries per CTA of the chunk kernel) against the oracle.
    The kv row of every third token is 4x the query of head (token mod 64): that head's logit on its own
    token, the last row of the query's last tile, is ~2^130 above the rest, so the running reference max is
    raised after earlier tiles were accumulated (the rescale of O and of the sums)."""
    cfg = csa_synth.CONFIGS[5].replace(ctx=8192 + 2, T=300)
    cap = (cfg.ctx + cfg.T) // cfg.ratio + 4
    run = G.Runner(cfg)
    host = csa_synth.synth_cache(cfg, cap)
    st_g = G.DevCache(host)
    ch = csa_synth.chunk_inputs(cfg)
    kv = ch.kv.clone()
    for i in range(0, cfg.T, 3):
        kv[i] = (4 * ch.q[i, i % cfg.H].float()).to(kv.dtype)
    ch = csa_synth.StepInputs(x=ch.x, q=ch.q, kv=kv, iq=ch.iq, iw=ch.iw)
    out, sel = run.prefill(st_g, ch, cfg.ctx)
    torch.cuda.synchronize()
    assert run.err.item() == 0
    _, n, _, ring, worst = _check_prefill(cfg, run, host, ch, out, sel, range(cfg.T), label="5' prefill T300 ctx8k")
    assert n == st_g.n_rows.item()
    G.check_pool_rows(st_g.window[0].cpu(), ring, "bf16", "window after chunk")
    print(f"prefill, every query: worst max-relative output error {worst:.2e}")


def test_gpu_decode_equals_gpu_prefill():
    """A chunk attended as one prefill call equals the same tokens decoded one at a time (Flash shapes,
    sparse regime, window eviction inside the chunk, 16 compress boundaries)."""
    cfg = csa_synth.CONFIGS[5].replace(ctx=8192 + 2, T=64)
    cap = (cfg.ctx + cfg.T) // 4 + 4
    host = csa_synth.synth_cache(cfg, cap)
    run = G.Runner(cfg)
    ch = csa_synth.chunk_inputs(cfg)
    st_p = G.DevCache(host)
    out_p, sel_p = run.prefill(st_p, ch, cfg.ctx)
    st_d = G.DevCache(host)
    outs = []
    for i in range(cfg.T):
        si = csa_synth.StepInputs(x=ch.x[:, i:i + 1], q=ch.q[i:i + 1], kv=ch.kv[i:i + 1], iq=ch.iq[i:i + 1],
                                  iw=ch.iw[i:i + 1])
        o, s, ns = run.decode_step(st_d, si)
        outs.append(o[0])
        assert sorted(s[0, :ns[0]].tolist()) == sorted(x for x in sel_p[i].tolist() if x >= 0), f"query {i}"
    torch.cuda.synchronize()
    assert run.err.item() == 0
    assert torch.equal(st_p.pool, st_d.pool) and torch.equal(st_p.ikeys, st_d.ikeys)
    assert torch.equal(st_p.window, st_d.window)
    assert torch.equal(st_p.front_attn, st_d.front_attn)
    G.check_rows(torch.stack(outs).cpu(), out_p.cpu(), "bf16", what="decode vs prefill", R=cfg.R)


@pytest.mark.parametrize("case", ["fresh_prompt", "tiny_prompt", "dense_to_sparse", "ratio128"])
def test_prefill_fresh_prompt_crossing_and_ratio128(case):
    """Prefill chunks beyond the long-cache workloads, every query checked against the oracle (selection, output
    rounded and un-rounded), with the rows the chunk emits and the window ring after it:
      * fresh_prompt: 300 tokens from an empty cache (pos0 = 0): the window fills during the chunk (queries 0-126
        see fewer than 128 window tokens) and every query is in the dense regime (at most 75 rows visible);
      * tiny_prompt: 7 tokens from an empty cache (one compressed row, fewer tokens than a 128-row tile);
      * dense_to_sparse: 400 tokens after 1900: the visible rows go from 475 to 575 and pass topk = 512 at
        query 151 (position 2051), inside the chunk;
      * ratio128: a ratio-128 layer (no indexer, every visible row attended), 300 tokens after 262044: a window
        of 128 tokens completes inside the chunk (row 2047 at position 262143)."""
    base = csa_synth.CONFIGS[5]
    if case == "fresh_prompt":
        cfg = base.replace(ctx=0, T=300)
    elif case == "tiny_prompt":
        cfg = base.replace(ctx=0, T=7)
    elif case == "dense_to_sparse":
        cfg = base.replace(ctx=1900, T=400)
    else:
        cfg = csa_synth.CONFIGS[4].replace(B=1, ctx=262144 - 100, T=300)
    cap = (cfg.ctx + cfg.T) // cfg.ratio + 4
    host = csa_synth.synth_cache(cfg, cap, B=1) if cfg.ctx else csa_synth.empty_cache(cfg, cap, B=1)
    run = G.Runner(cfg)
    st_g = G.DevCache(host)
    ch = csa_synth.chunk_inputs(cfg)
    out, sel = run.prefill(st_g, ch, cfg.ctx)
    torch.cuda.synchronize()
    assert run.err.item() == 0
    if case == "ratio128":
        queries = sorted(set(range(0, cfg.T, 3)) | {cfg.T - 1, 98, 99, 100, 227, 228})
    else:
        queries = range(cfg.T)
    st, n, lo, ring, worst = G.check_prefill_chunk(cfg, run, host, ch, out, sel, queries,
                                                   label=f"prefill {case} (T {cfg.T}, ctx {cfg.ctx}, ratio {cfg.ratio})")
    assert n == st_g.n_rows.item() == (cfg.ctx + cfg.T) // cfg.ratio
    G.check_pool_rows(st_g.pool[0, lo:n].cpu(), st["pool"][0, lo:n], "bf16", "chunk pool rows", R=cfg.R)
    if cfg.has_indexer:
        G.check_pool_rows(st_g.ikeys[0, lo:n].cpu(), st["ikeys"][0, lo:n], "bf16", "chunk index rows", R=cfg.R)
        nvis = [O.visible_rows(oracle_layer(cfg), n, cfg.ctx + i) for i in range(cfg.T)]
        dense = [i for i in range(cfg.T) if nvis[i] <= cfg.topk]
        g_sel = sel.cpu()
        for i in dense:  # the dense regime selects every visible row, padded with -1
            assert g_sel[i, :nvis[i]].tolist() == list(range(nvis[i])) and (g_sel[i, nvis[i]:] == -1).all()
    G.check_pool_rows(st_g.window[0].cpu(), ring, "bf16", "window after chunk")
    print(f"prefill {case}: worst max-relative output error {worst:.2e}")


def test_config5_chunk_equals_4096_decode_steps():
    """Config 5 in full: the 4096-token chunk on the 65536-token cache as one prefill call, against the same
    tokens decoded one at a time on the GPU (4096 decode steps through the four calls).

    The two paths project the chunk's tokens with different fp32 summation orders along the hidden axis (one
    token: split-K partials summed in split order; a 4096-token chunk: one accumulation per tile), so a few
    projections round to neighbouring bf16 values and the pools need not be bit-identical.  Each path is held to
    the rules of the other tests instead: its projections against the oracle's, its emitted rows against the
    oracle pooling its own projections.  The window ring and row counts must be identical.  Where the two
    selections of a query are the same set, the two outputs must agree within twice the output rule (each is
    held to the rule against the oracle, and their pools may differ by those rounding flips); where they
    differ, each set must pass the gap rule against the oracle's scores over its own path's index keys.  Both
    paths' outputs of those queries and of 48 spread queries are checked against the oracle recomputed with
    their own set and rows."""
    cfg = csa_synth.CONFIGS[5]
    cap = (cfg.ctx + cfg.T) // cfg.ratio + 4
    host = csa_synth.synth_cache(cfg, cap)
    run = G.Runner(cfg)
    ch = csa_synth.chunk_inputs(cfg)
    st_p = G.DevCache(host)
    out_p, sel_p = run.prefill(st_p, ch, cfg.ctx)
    proj_p = {k: v.cpu() for k, v in run.projs.items()}
    st_d = G.DevCache(host)
    out_d = torch.empty_like(out_p)
    sel_d = torch.full_like(sel_p, -1)
    proj_d = {"attn": [], "index": []}
    for i in range(cfg.T):
        si = csa_synth.StepInputs(x=ch.x[:, i:i + 1], q=ch.q[i:i + 1], kv=ch.kv[i:i + 1], iq=ch.iq[i:i + 1],
                                  iw=ch.iw[i:i + 1])
        o, s, ns = run.decode_step(st_d, si)
        out_d[i] = o[0]
        sel_d[i] = s[0]
        for k in proj_d:
            proj_d[k].append(run.projs[k])
    torch.cuda.synchronize()
    assert run.err.item() == 0
    assert torch.equal(st_p.window, st_d.window)
    assert torch.equal(st_p.n_rows, st_d.n_rows)
    proj_d = {k: torch.cat(v, dim=1).cpu() for k, v in proj_d.items()}
    layer = oracle_layer(cfg)
    invf = f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    sink = f64(csa_synth.sinks(cfg))
    ca, ci = oracle_comp(run.ca_host), oracle_comp(run.ci_host)
    x = f64(ch.x)
    n = st_p.n_rows.item()
    lo = cfg.ctx // cfg.ratio
    keys_of = {}
    for name, st_g, pr in (("prefill", st_p, proj_p), ("decode", st_d, proj_d)):
        o = _oracle_seq_state(host, 0)
        n0 = o["n_rows"].copy()
        _, pool_o, _, _ = G.oracle_compress_checked(layer, ca, x, o["pos"], o["front_a"], o["pool"], n0, invf,
                                                    pr["attn"], f"{name} attn")
        _, ik_o, _, _ = G.oracle_compress_checked(layer, ci, x, o["pos"], o["front_i"], o["ikeys"], n0, invf,
                                                  pr["index"], f"{name} index")
        G.check_pool_rows(st_g.pool[0, lo:n].cpu(), pool_o[0, lo:n], "bf16", f"{name} pool rows", R=cfg.R)
        G.check_pool_rows(st_g.ikeys[0, lo:n].cpu(), ik_o[0, lo:n], "bf16", f"{name} index rows", R=cfg.R)
        keys_of[name] = (f64(st_g.pool[0].cpu()), f64(st_g.ikeys[0].cpu()))
    same_pool = bool(torch.equal(st_p.pool, st_d.pool) and torch.equal(st_p.ikeys, st_d.ikeys))
    sp, sd = torch.sort(sel_p, dim=1).values, torch.sort(sel_d, dim=1).values
    assert (sp >= 0).all() and (sd >= 0).all()  # 16384+ rows visible: sparse throughout
    same = (sp == sd).all(dim=1).cpu()
    idx_same = torch.nonzero(same).flatten()
    for k in range(0, len(idx_same), 256):
        blk = idx_same[k:k + 256].to("cuda")
        G.check_rows(out_p[blk].cpu(), out_d[blk].cpu(), "bf16", what="decode vs prefill", R=cfg.R, scale=2.0)
    differ = torch.nonzero(~same).flatten().tolist()
    n_pool_diff = int((st_p.pool != st_d.pool).sum().item() + (st_p.ikeys != st_d.ikeys).sum().item())
    print(f"config 5 decode == prefill: pools identical: {same_pool} ({n_pool_diff} elements differ); "
          f"{len(idx_same)} of {cfg.T} selections identical, {len(differ)} differ")
    assert len(differ) <= cfg.T // 16, f"{len(differ)} queries selected different sets"
    window0 = f64(host.window[0])
    kvr = [O.store(O.rope(f64(ch.kv[i]), cfg.ctx + i, invf), "bf16") for i in range(cfg.T)]
    sample = sorted(set(differ) | set(range(0, cfg.T, cfg.T // 48)) | {cfg.T - 1})
    for i in sample:
        p = cfg.ctx + i
        nv = O.visible_rows(layer, n, p)
        win = [window0[t % cfg.W] if t < cfg.ctx else kvr[t - cfg.ctx] for t in O.window_tokens(layer, p)]
        qr = O.store(O.rope(f64(ch.q[i]), p, invf), "bf16")
        for name, s_, o_ in (("prefill", sel_p, out_p), ("decode", sel_d, out_d)):
            pool, ikeys = keys_of[name]
            rows = s_[i].cpu().numpy()
            if i in differ:
                scores = O.index_scores(layer, f64(ch.iq[i]), f64(ch.iw[i]), ikeys[:nv], p, invf)
                G.check_topk(rows, scores, cfg.topk, nv, what=f"{name} query {i} top-k")
            keys = np.concatenate([pool[np.sort(rows)], np.stack(win)])
            o = O.attend(layer, qr, keys, sink)
            G.check_rows(o_[i].cpu(), O.output_rows(layer, o, p, invf), "bf16", what=f"{name} query {i}",
                         R=cfg.R, exact=G.exact_output(o, p, invf), label=f"5 {name} path, full-chunk sample")


def test_config3_every_sequence_four_steps():
    """Config 3 at full size with every one of the 32 sequences checked against the oracle for four decode steps
    (projections, selection under the gap rule, output rounded and un-rounded, emitted rows).  The GPU runs
    first; the oracle then follows one sequence at a time, so only one sequence's float64 state is held."""
    cfg = csa_synth.CONFIGS[3]
    steps = 4  # the fourth token (position 32771) completes a window: one row emitted per sequence
    cap = cfg.ctx // cfg.ratio + 8
    host = csa_synth.synth_cache(cfg, cap)
    run = G.Runner(cfg)
    st_g = G.DevCache(host)
    rec = []
    for step in range(steps):
        si = csa_synth.step_inputs(cfg, step)
        out, sel, n_sel = run.decode_step(st_g, si)
        torch.cuda.synchronize()
        rec.append((si, out.cpu(), sel.cpu().numpy(), n_sel.cpu().numpy(),
                    {k: v.cpu() for k, v in run.projs.items()}))
    assert run.err.item() == 0
    layer = oracle_layer(cfg)
    ca, ci = oracle_comp(run.ca_host), oracle_comp(run.ci_host)
    sink, invf = f64(csa_synth.sinks(cfg)), f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    pool_g = st_g.pool.cpu()
    for b in range(cfg.B):
        st_o = _oracle_seq_state(host, b)
        for step, (si, out, sel, n_sel, projs) in enumerate(rec):
            _oracle_decode_check(layer, ca, ci, st_o, _step_rows(si, b), sink, invf, out[b], sel[b], n_sel[b],
                                 f"seq {b} step {step}", {k: v[b:b + 1] for k, v in projs.items()},
                                 label=f"3 {cfg.name}")
        lo, n = cfg.ctx // cfg.ratio, int(st_o["n_rows"][0])
        G.check_pool_rows(pool_g[b, lo:n], st_o["pool"][0, lo:n], "bf16", f"seq {b} new pool rows", R=cfg.R)


def _ragged_cache(cfg, cap, ctxs):
    host = csa_synth.synth_cache(cfg, cap, B=len(ctxs), ctx=max(ctxs))
    for b, c in enumerate(ctxs):
        n = c // cfg.ratio
        host.pool[b, n:] = 0
        if host.ikeys is not None:
            host.ikeys[b, n:] = 0
        host.n_rows[b] = n
        host.pos[b] = c
    return host


@pytest.mark.parametrize("overlap", [False, True, "one_stream"],
                         ids=["serial", "overlapped_indexer", "overlapped_one_stream"])
def test_ragged_batch_edges(overlap):
    """One batch mixing an empty cache, a cache shorter than the window, the dense/sparse threshold
    (n_vis == topk and topk + 1) and a long cache; with csa_index_topk, with csa_index_topk_overlapped
    scanning while the index pool's compress call runs on another stream, and with the pair call followed by
    csa_index_topk_overlapped on one stream (some steps emit a row)."""
    cfg = csa_synth.CONFIGS[3].replace(B=6)
    ctxs = [0, 3, 100, 2047, 2051, 9000]
    cap = max(ctxs) // 4 + 8
    host = _ragged_cache(cfg, cap, ctxs)
    run = G.Runner(cfg)
    st_g = G.DevCache(host)
    layer = oracle_layer(cfg)
    ca, ci = oracle_comp(run.ca_host), oracle_comp(run.ci_host)
    sink, invf = f64(csa_synth.sinks(cfg)), f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    st_o = {b: _oracle_seq_state(host, b) for b in range(len(ctxs))}
    for step in range(5):
        si = csa_synth.step_inputs(cfg, step, B=len(ctxs))
        out, sel, n_sel = run.decode_step(st_g, si, overlap=overlap)
        torch.cuda.synchronize()
        for b in range(len(ctxs)):
            _oracle_decode_check(layer, ca, ci, st_o[b], _step_rows(si, b), sink, invf, out[b].cpu(),
                                 sel[b].cpu().numpy(), n_sel[b].item(), f"ctx {ctxs[b]} step {step}",
                                 _seq_projs(run, b))
    assert run.err.item() == 0
    assert n_sel.cpu().tolist()[3] == 512  # 2047 + 5 tokens -> 513 rows visible: sparse, 512 kept


def test_decode_without_selection_attends_every_visible_row():
    """A layer with an indexer called without a selection attends to every visible row: up to 1300 rows per
    query here, more than the workspace's splits can hold in 160-row chunks, so the multi-tile kernel serves
    it.  Checked against the oracle's attention over all visible rows."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=3)
    ctxs = [1000, 3001, 5202]
    cap = max(ctxs) // 4 + 8
    host = _ragged_cache(cfg, cap, ctxs)
    run = G.Runner(cfg)
    st_g = G.DevCache(host)
    layer = oracle_layer(cfg)
    st_o = oracle_state(host)
    sink, invf = f64(csa_synth.sinks(cfg)), f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    si = csa_synth.step_inputs(cfg, 0, B=len(ctxs))
    out = torch.empty(len(ctxs), cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
    csa.attend_decode(run.L, G.dev(si.q), G.dev(si.kv), run.sink, st_g.window, st_g.pool, st_g.n_rows, None, None,
                      st_g.pos, run.inv_freq, out, err=run.err)
    ref, window, err = O.attend_decode(layer, f64(si.q), f64(si.kv), sink, st_o["window"], st_o["pool"],
                                       st_o["n_rows"], None, None, st_o["pos"], invf)
    torch.cuda.synchronize()
    assert err == 0 and run.err.item() == 0
    for b in range(len(ctxs)):
        G.check_rows(out[b].cpu(), ref[b], layer.dtype, what=f"ctx {ctxs[b]} output", R=layer.R)
        G.check_pool_rows(st_g.window[b].cpu(), window[b], "bf16", "window")  # the new token's ring slot


def test_topk_ties_go_to_lower_rows():
    """All index keys equal -> all scores tie exactly; the selection must be rows 0 .. topk-1."""
    cfg = csa_synth.CONFIGS[3].replace(B=2)
    cap = 1200
    host = _ragged_cache(cfg, cap, [4000, 4400])
    host.ikeys[:, :] = host.ikeys[:, :1].clone()
    run = G.Runner(cfg)
    st_g = G.DevCache(host)
    si = csa_synth.step_inputs(cfg, 0, B=2)
    _, sel, n_sel = run.decode_step(st_g, si)
    torch.cuda.synchronize()
    for b in range(2):
        assert n_sel[b].item() == 512
        assert sel[b].tolist() == list(range(512))


def test_compress_chunking_invariance_gpu():
    """Any split of the same tokens into compress calls gives bit-identical pools and frontiers."""
    cfg = csa_synth.CONFIGS[2].replace(B=2)
    cap = 64
    xs = csa_synth.hidden(cfg, 77, B=2)
    run = G.Runner(cfg)
    results = []
    for splits in ([77], [1] * 77, [3, 5, 8, 61], [13, 64]):
        st = G.DevCache(csa_synth.empty_cache(cfg, cap, B=2))
        p = 0
        for s in splits:
            run.compress(st, xs[:, p:p + s])
            st.pos += s
            p += s
        torch.cuda.synchronize()
        results.append(st)
    for st in results[1:]:
        assert torch.equal(st.pool, results[0].pool) and torch.equal(st.ikeys, results[0].ikeys)
        assert torch.equal(st.front_attn, results[0].front_attn)
        assert torch.equal(st.n_rows, results[0].n_rows)
    assert run.err.item() == 0


def test_device_errors_fail_closed():
    """Inconsistent state, capacity overflow and out-of-range selections raise error bits and leave the
    affected state untouched."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[2].replace(B=2)
    run = G.Runner(cfg)
    # state: n_rows inconsistent with pos for sequence 0
    st = G.DevCache(_ragged_cache(cfg, 40, [40, 40]))
    st.n_rows[0] = 3
    before = st.pool.clone(), st.front_attn.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa.compress_append(run.L, run.ca, G.dev(csa_synth.hidden(cfg, 8, B=2)), st.pos, st.front_attn, st.pool,
                        st.n_rows, run.inv_freq, err=err)
    torch.cuda.synchronize()
    assert err.item() == csa.DEV_STATE
    assert torch.equal(st.pool[0], before[0][0]) and torch.equal(st.front_attn[0], before[1][0])
    assert st.n_rows.tolist() == [3, 12]
    # capacity: 40 tokens fill 10 rows of a 10-row pool; 4 more would emit row 10
    st = G.DevCache(_ragged_cache(cfg, 10, [36, 40]))
    err.zero_()
    before = st.pool.clone()
    csa.compress_append(run.L, run.ca, G.dev(csa_synth.hidden(cfg, 4, B=2)), st.pos, st.front_attn, st.pool,
                        st.n_rows, run.inv_freq, err=err)
    torch.cuda.synchronize()
    assert err.item() == csa.DEV_CAPACITY
    assert st.n_rows.tolist() == [10, 10] and torch.equal(st.pool[1], before[1])
    # out-of-range selection
    st = G.DevCache(_ragged_cache(cfg, 40, [100, 100]))
    err.zero_()
    si = csa_synth.step_inputs(cfg, 0, B=2)
    sel = torch.full((2, cfg.topk), -1, dtype=torch.int32, device="cuda")
    sel[:, 0] = 5
    sel[1, 1] = 30  # only 25 rows exist
    n_sel = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    out = torch.empty(2, cfg.H, cfg.D, dtype=torch.bfloat16, device="cuda")
    csa.attend_decode(run.L, G.dev(si.q), G.dev(si.kv), run.sink, st.window, st.pool, st.n_rows, sel, n_sel, st.pos,
                      run.inv_freq, out, err=err)
    torch.cuda.synchronize()
    assert err.item() == csa.DEV_RANGE
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("B,ctx,steps", [(8, 8192 + 1, 6), (32, 32768 + 2, 4)])
def test_compress_pair_single_tokens_against_oracle(B, ctx, steps):
    """csa_compress_append_pair, one token per sequence (both projections in one grid, both pooling steps in
    one launch), across window completions: each pool's projections and emitted rows against the oracle on
    sampled sequences (the same rules as the single call); a sequence with an inconsistent row count is refused
    and left unchanged."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=B, ctx=ctx)
    cap = (ctx + steps) // 4 + 8
    host = csa_synth.synth_cache(cfg, cap, B=B)
    run = G.Runner(cfg)
    st = G.DevCache(host)
    st.n_rows[B - 1] -= 3  # state error for the last sequence (its positions only grow: it stays inconsistent)
    ni = st.n_rows.clone()
    bad_before = (st.pool[B - 1].clone(), st.ikeys[B - 1].clone(), st.front_attn[B - 1].clone())
    layer = oracle_layer(cfg)
    ca, ci = oracle_comp(run.ca_host), oracle_comp(run.ci_host)
    invf = f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    seqs = [0, B // 2, B - 2]
    full = oracle_state(host)
    st_o = {b: {k: None if v is None else v[b:b + 1].copy() for k, v in full.items()} for b in seqs}
    del full
    F = st.front_attn.shape[1]
    for step in range(steps):
        x = csa_synth.hidden(cfg, 1, B=B, tag=100 + step)
        slots = st.pos.long() % F
        csa.compress_append_pair(run.L, run.ca, run.ci, G.dev(x), st.pos, st.front_attn, st.pool, st.n_rows,
                                 st.front_index, st.ikeys, ni, run.inv_freq, err=run.err)
        torch.cuda.synchronize()
        for b in seqs:
            o = st_o[b]
            xb = f64(x[b:b + 1])
            n0 = o["n_rows"].copy()
            pa = st.front_attn[b, slots[b]].view(1, 1, -1).cpu()
            pi = st.front_index[b, slots[b]].view(1, 1, -1).cpu()
            o["front_a"], o["pool"], n_a, e1 = G.oracle_compress_checked(layer, ca, xb, o["pos"], o["front_a"], o["pool"],
                                                                         n0, invf, pa, f"seq {b} step {step} attn")
            o["front_i"], o["ikeys"], n_i, e2 = G.oracle_compress_checked(layer, ci, xb, o["pos"], o["front_i"],
                                                                          o["ikeys"], n0, invf, pi,
                                                                          f"seq {b} step {step} index")
            assert e1 == 0 and e2 == 0
            o["n_rows"], o["pos"] = n_a, o["pos"] + 1
        st.pos += 1
    assert run.err.item() == csa.DEV_STATE
    assert torch.equal(st.n_rows, ni)
    for b in seqs:
        o = st_o[b]
        n = int(o["n_rows"][0])
        assert n == st.n_rows[b].item()
        lo = ctx // cfg.ratio
        G.check_pool_rows(st.pool[b, lo:n].cpu(), o["pool"][0, lo:n], "bf16", f"seq {b} pool rows", R=cfg.R)
        G.check_pool_rows(st.ikeys[b, lo:n].cpu(), o["ikeys"][0, lo:n], "bf16", f"seq {b} index rows", R=cfg.R)
    assert torch.equal(st.pool[B - 1], bad_before[0]) and torch.equal(st.ikeys[B - 1], bad_before[1])
    assert torch.equal(st.front_attn[B - 1], bad_before[2])
    assert st.n_rows[B - 1].item() == host.n_rows[B - 1].item() - 3


def test_compress_pair_chunk_equals_two_calls():
    """A chunk (T > 1) through csa_compress_append_pair is the two single calls in turn: identical results."""
    import deepseek_v4_compressed_csa_gb300 as csa
    B, ctx, T = 3, 4096 + 3, 6
    cfg = csa_synth.CONFIGS[3].replace(B=B, ctx=ctx)
    host = csa_synth.synth_cache(cfg, (ctx + T) // 4 + 8, B=B)
    run = G.Runner(cfg)
    one, two = G.DevCache(host), G.DevCache(host)
    ni_one, ni_two = one.n_rows.clone(), two.n_rows.clone()
    x = G.dev(csa_synth.hidden(cfg, T, B=B, tag=7))
    e1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    e2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa.compress_append(run.L, run.ca, x, one.pos, one.front_attn, one.pool, one.n_rows, run.inv_freq, err=e1)
    csa.compress_append(run.L, run.ci, x, one.pos, one.front_index, one.ikeys, ni_one, run.inv_freq, err=e1)
    csa.compress_append_pair(run.L, run.ca, run.ci, x, two.pos, two.front_attn, two.pool, two.n_rows,
                             two.front_index, two.ikeys, ni_two, run.inv_freq, err=e2)
    torch.cuda.synchronize()
    assert e1.item() == e2.item() == 0
    assert torch.equal(one.pool, two.pool) and torch.equal(one.ikeys, two.ikeys)
    assert torch.equal(one.front_attn, two.front_attn) and torch.equal(one.front_index, two.front_index)
    assert torch.equal(one.n_rows, two.n_rows) and torch.equal(ni_one, ni_two)


def test_advance_positions():
    """csa_advance_positions adds `by` to every position (more sequences than one block holds), and leaves the
    array alone for B = 0."""
    import deepseek_v4_compressed_csa_gb300 as csa
    pos = torch.arange(300, dtype=torch.int32, device="cuda") * 7 - 5
    want = pos.clone() + 3
    csa.advance_positions(pos, 3)
    csa.advance_positions(pos[:0], 9)
    torch.cuda.synchronize()
    assert torch.equal(pos, want)


def test_host_validation_raises():
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[2].replace(B=1)
    run = G.Runner(cfg)
    st = G.DevCache(csa_synth.empty_cache(cfg, 8, B=1))
    x = G.dev(csa_synth.hidden(cfg, 4, B=1))
    bad = csa.Layer(**{**vars(run.L), "D": 500})
    with pytest.raises(csa.CSAError) as ei:
        csa.compress_append(bad, run.ca, x, st.pos, st.front_attn, st.pool, st.n_rows, run.inv_freq)
    assert ei.value.code == 1
    tiny_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(csa.CSAError) as ei:
        csa.compress_append(run.L, run.ca, x, st.pos, st.front_attn, st.pool, st.n_rows, run.inv_freq, ws=tiny_ws)
    assert ei.value.code == 4


def test_binding_rejects_wrong_dtype_and_shape_before_any_launch():
    """On the device too: an fp32 query handed to a bf16 layer, or a selection of the wrong width, raises in the
    binding and enqueues nothing (the library's launch count and the outputs stay as they were)."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=2)
    run = G.Runner(cfg)
    st = G.DevCache(_ragged_cache(cfg, 40, [100, 100]))
    si = csa_synth.step_inputs(cfg, 0, B=2)
    sel = torch.zeros(2, cfg.topk, dtype=torch.int32, device="cuda")
    n_sel = torch.ones(2, dtype=torch.int32, device="cuda")
    out = torch.full((2, cfg.H, cfg.D), 7.0, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    before = csa.kernel_launches()
    with pytest.raises(TypeError, match="q"):
        csa.attend_decode(run.L, G.dev(si.q).float(), G.dev(si.kv), run.sink, st.window, st.pool, st.n_rows, sel,
                          n_sel, st.pos, run.inv_freq, out, err=run.err)
    with pytest.raises(ValueError, match="sel"):
        csa.attend_decode(run.L, G.dev(si.q), G.dev(si.kv), run.sink, st.window, st.pool, st.n_rows, sel[:, :100],
                          n_sel, st.pos, run.inv_freq, out, err=run.err)
    with pytest.raises(TypeError, match="iw"):
        csa.index_topk(run.L, G.dev(si.iq), G.dev(si.iw).float(), st.ikeys, st.n_rows, st.pos, run.inv_freq, sel,
                       n_sel, err=run.err)
    torch.cuda.synchronize()
    assert csa.kernel_launches() == before
    assert (out == 7.0).all() and run.err.item() == 0
