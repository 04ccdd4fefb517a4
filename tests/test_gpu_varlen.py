"""Packed variable-length prefill batches (csa_compress_append_varlen, csa_attend_prefill_varlen) on the GPU.

A batch of chunks of different lengths at different positions, packed back to back, must give every sequence
what a prefill chunk of its own gives ("DeepSeek-V4-Flash: native deepseek_v4 AR backend", MTPLX #216,
"Verification": decode == prefill across chunked prefill and batching).  Each sequence is checked against the
oracle's chunk from the GPU's own projections of it (selection under the gap rule, outputs rounded and
un-rounded, the rows it emits, the window ring after it); an empty chunk leaves its sequence untouched.
"""
import numpy as np
import pytest
import torch

import csa_synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests import _gpu as G

# (context before the chunk, chunk length): a fresh prompt; the dense->sparse threshold (position 2051) inside the
# chunk; a single token; an empty chunk; a chunk whose later queries' windows lie wholly inside it
SPECS = [(0, 300), (1990, 100), (9001, 1), (5003, 0), (4097, 160)]


def _seq_cache(cfg, cap, b, ctx):
    c = cfg.replace(cid=cfg.cid + 40 + b)  # each sequence its own random stream
    return csa_synth.synth_cache(c, cap, B=1, ctx=ctx) if ctx else csa_synth.empty_cache(c, cap, B=1)


def _packed(chunks, field):
    return torch.cat([getattr(ch, field) if field != "x" else ch.x[0] for ch in chunks])


def test_varlen_prefill_batch_against_oracle():
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[5]
    B = len(SPECS)
    cap = max(c + t for c, t in SPECS) // cfg.ratio + 8
    parts = [_seq_cache(cfg, cap, b, c) for b, (c, _) in enumerate(SPECS)]
    cat = lambda k: None if getattr(parts[0], k) is None else torch.cat([getattr(p, k) for p in parts])  # noqa: E731
    host = csa_synth.Cache(**{k: cat(k) for k in vars(parts[0])})
    chunks = [csa_synth.chunk_inputs(cfg.replace(cid=cfg.cid + 80 + b), t) for b, (_, t) in enumerate(SPECS)]
    lens = [t for _, t in SPECS]
    N, T_max = sum(lens), max(lens)
    cu_host = [0] + np.cumsum(lens).tolist()
    run = G.Runner(cfg)
    st = G.DevCache(host)
    cu = torch.tensor(cu_host, dtype=torch.int32, device="cuda")
    x = G.dev(_packed(chunks, "x"))
    projs = {}
    n_i = st.n_rows.clone()
    for name, comp, front, pool, n in (("attn", run.ca, st.front_attn, st.pool, st.n_rows),
                                       ("index", run.ci, st.front_index, st.ikeys, n_i)):
        ws = torch.zeros(csa.workspace_size(run.L, csa.OP_COMPRESS_VARLEN, B, N, cap), dtype=torch.uint8,
                         device="cuda")
        csa.compress_append_varlen(run.L, comp, x, cu, T_max, st.pos, front, pool, n, run.inv_freq, ws=ws,
                                   err=run.err)
        width = 2 * cfg.lanes * comp.d
        off = (4 * B + 255) // 256 * 256  # workspace layout: [B] int32 flags, then [N, 2*L*d] projections
        projs[name] = ws[off:off + N * width * 2].view(cfg.storage).view(N, width).clone()
    out = torch.empty(N, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
    sel = torch.empty(N, cfg.topk, dtype=torch.int32, device="cuda")
    csa.attend_prefill_varlen(run.L, G.dev(_packed(chunks, "q")), G.dev(_packed(chunks, "kv")),
                              G.dev(_packed(chunks, "iq")), G.dev(_packed(chunks, "iw")), run.sink, cu, T_max, st.pos,
                              st.window, st.pool, st.ikeys, st.n_rows, run.inv_freq, out, sel_out=sel, err=run.err)
    torch.cuda.synchronize()
    assert run.err.item() == 0
    assert torch.equal(n_i, st.n_rows)
    for b, (ctx, T) in enumerate(SPECS):
        lo_b, hi_b = cu_host[b], cu_host[b + 1]
        if T == 0:
            assert st.n_rows[b].item() == host.n_rows[b].item()
            for k in ("pool", "ikeys", "window", "front_attn", "front_index"):
                assert torch.equal(getattr(st, k)[b].cpu(), getattr(host, k)[b]), f"empty chunk changed {k}"
            continue
        cfg_b = cfg.replace(ctx=ctx, T=T)
        run.projs = {k: v[lo_b:hi_b][None].cpu() for k, v in projs.items()}
        queries = range(T) if T <= 160 else sorted(set(range(0, T, 4)) | {T - 1, 126, 127, 128, 129})
        st_o, n, lo, ring, worst = G.check_prefill_chunk(cfg_b, run, parts[b], chunks[b], out[lo_b:hi_b],
                                                         sel[lo_b:hi_b], queries,
                                                         label=f"varlen prefill batch (B {B}, N {N})")
        assert n == st.n_rows[b].item() == (ctx + T) // cfg.ratio, f"seq {b} rows"
        G.check_pool_rows(st.pool[b, lo:n].cpu(), st_o["pool"][0, lo:n], "bf16", f"seq {b} pool rows", R=cfg.R)
        G.check_pool_rows(st.ikeys[b, lo:n].cpu(), st_o["ikeys"][0, lo:n], "bf16", f"seq {b} index rows", R=cfg.R)
        G.check_pool_rows(st.window[b].cpu(), ring, "bf16", f"seq {b} window after chunk")


def test_varlen_sizes_refused_on_host():
    """Packed sizes the host can see are checked before anything is enqueued."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[5]
    run = G.Runner(cfg)
    cap = 64
    st = G.DevCache(csa_synth.empty_cache(cfg, cap, B=2))
    cu = torch.tensor([0, 3, 5], dtype=torch.int32, device="cuda")
    x = torch.zeros(5, cfg.X, dtype=cfg.storage, device="cuda")
    with pytest.raises(ValueError):  # T_max beyond N
        csa.compress_append_varlen(run.L, run.ca, x, cu, 6, st.pos, st.front_attn, st.pool, st.n_rows, run.inv_freq)
    with pytest.raises(ValueError):  # a row table of the wrong length
        csa.compress_append_varlen(run.L, run.ca, x, cu[:2], 3, st.pos, st.front_attn, st.pool, st.n_rows,
                                   run.inv_freq)


def test_varlen_inconsistent_row_table_is_flagged():
    """A row-table entry that ends before it starts is flagged CSA_DEV_STATE by the compress call, which leaves that
    sequence unchanged; the other sequences (even overlapping rows) are processed, and every row index the
    attention call derives from the table stays inside the packed buffers."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[5]
    B, N, cap = 3, 8, 1100
    parts = [_seq_cache(cfg, cap, b, 4000 + 4 * b) for b in range(B)]
    host = csa_synth.Cache(**{k: None if getattr(parts[0], k) is None else torch.cat([getattr(p, k) for p in parts])
                              for k in vars(parts[0])})
    run = G.Runner(cfg)
    st = G.DevCache(host)
    cu = torch.tensor([0, 5, 3, 8], dtype=torch.int32, device="cuda")
    ch = csa_synth.chunk_inputs(cfg.replace(cid=cfg.cid + 90), N)
    n_i = st.n_rows.clone()
    csa.compress_append_varlen(run.L, run.ca, G.dev(ch.x[0]), cu, 5, st.pos, st.front_attn, st.pool, st.n_rows,
                               run.inv_freq, err=run.err)
    csa.compress_append_varlen(run.L, run.ci, G.dev(ch.x[0]), cu, 5, st.pos, st.front_index, st.ikeys, n_i,
                               run.inv_freq, err=run.err)
    out = torch.empty(N, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
    csa.attend_prefill_varlen(run.L, G.dev(ch.q), G.dev(ch.kv), G.dev(ch.iq), G.dev(ch.iw), run.sink, cu, 5, st.pos,
                              st.window, st.pool, st.ikeys, st.n_rows, run.inv_freq, out, err=run.err)
    torch.cuda.synchronize()
    assert run.err.item() & csa.DEV_STATE
    assert st.n_rows.tolist() == [(4000 + 5) // 4, host.n_rows[1].item(), (4008 + 5) // 4]
    for k in ("pool", "window", "front_attn"):
        assert torch.equal(getattr(st, k)[1].cpu(), getattr(host, k)[1]), f"flagged sequence changed {k}"


def test_varlen_prefill_ratio128_without_indexer():
    """The same on a ratio-128 layer (no indexer: every visible row attended): a fresh prompt whose chunk completes
    row 0, a short chunk, and a chunk that completes row 2047 (position 262143)."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[4].replace(B=1)
    specs = [(0, 130), (1000, 50), (262144 - 100, 300)]
    B = len(specs)
    cap = max(c + t for c, t in specs) // cfg.ratio + 4
    parts = [_seq_cache(cfg, cap, b, c) for b, (c, _) in enumerate(specs)]
    host = csa_synth.Cache(**{k: None if getattr(parts[0], k) is None else torch.cat([getattr(p, k) for p in parts])
                              for k in vars(parts[0])})
    chunks = [csa_synth.chunk_inputs(cfg.replace(cid=cfg.cid + 80 + b), t) for b, (_, t) in enumerate(specs)]
    lens = [t for _, t in specs]
    N, T_max = sum(lens), max(lens)
    cu_host = [0] + np.cumsum(lens).tolist()
    run = G.Runner(cfg)
    st = G.DevCache(host)
    cu = torch.tensor(cu_host, dtype=torch.int32, device="cuda")
    ws = torch.zeros(csa.workspace_size(run.L, csa.OP_COMPRESS_VARLEN, B, N, cap), dtype=torch.uint8, device="cuda")
    csa.compress_append_varlen(run.L, run.ca, G.dev(_packed(chunks, "x")), cu, T_max, st.pos, st.front_attn,
                               st.pool, st.n_rows, run.inv_freq, ws=ws, err=run.err)
    width = 2 * cfg.lanes * cfg.D
    off = (4 * B + 255) // 256 * 256
    proj = ws[off:off + N * width * 2].view(cfg.storage).view(N, width).clone()
    out = torch.empty(N, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
    sel = torch.empty(N, cfg.topk, dtype=torch.int32, device="cuda")
    csa.attend_prefill_varlen(run.L, G.dev(_packed(chunks, "q")), G.dev(_packed(chunks, "kv")), None, None,
                              run.sink, cu, T_max, st.pos, st.window, st.pool, None, st.n_rows, run.inv_freq, out,
                              sel_out=sel, err=run.err)
    torch.cuda.synchronize()
    assert run.err.item() == 0
    for b, (ctx, T) in enumerate(specs):
        lo_b, hi_b = cu_host[b], cu_host[b + 1]
        run.projs = {"attn": proj[lo_b:hi_b][None].cpu()}
        queries = range(T) if T <= 130 else sorted(set(range(0, T, 3)) | {T - 1, 98, 99, 100, 227, 228})
        st_o, n, lo, ring, worst = G.check_prefill_chunk(cfg.replace(ctx=ctx, T=T), run, parts[b], chunks[b],
                                                         out[lo_b:hi_b], sel[lo_b:hi_b], queries,
                                                         label=f"varlen prefill batch, ratio 128 (B {B})")
        assert n == st.n_rows[b].item() == (ctx + T) // cfg.ratio, f"seq {b} rows"
        G.check_pool_rows(st.pool[b, lo:n].cpu(), st_o["pool"][0, lo:n], "bf16", f"seq {b} pool rows", R=cfg.R)
        G.check_pool_rows(st.window[b].cpu(), ring, "bf16", f"seq {b} window after chunk")
