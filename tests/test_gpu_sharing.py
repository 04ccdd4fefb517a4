"""Cross-layer sharing (DeepSeek-V4.1, "deepseek-v41-mlx" README, "Cross-layer sharing") on the GPU.

A layer that owns no compressor calls only csa_index_topk (an index-source layer: its own queries against the
owner's index keys) and csa_attend_decode (its own queries, sinks and window ring, the owner's compressed rows),
or only csa_attend_decode with the owner's selection of the same step.  Checked against the oracle's consumer step
on sampled sequences, every step, with the owner checked as in the decode tests; the consumers must leave the
owner's caches untouched.
"""
import numpy as np
import pytest
import torch

import csa_synth
from oracle import csa_oracle as O
from tests._common import f64, oracle_comp, oracle_layer

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests import _gpu as G
    from tests.test_gpu_parity import _oracle_decode_check, _oracle_seq_state, _seq_projs, _step_rows


def test_owner_with_index_source_and_plain_consumers():
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=8, ctx=9001)
    steps, seqs = 6, (0, 5)
    cap = cfg.ctx // 4 + 8
    host = csa_synth.synth_cache(cfg, cap)
    run = G.Runner(cfg)
    st = G.DevCache(host)
    # two consumer layers: their own sinks, inputs and window rings (other seeded streams)
    cons = []
    for k in (1, 2):
        c = cfg.replace(cid=cfg.cid + 600 + k)
        win = csa_synth.synth_cache(c, cap, B=cfg.B).window
        cons.append(dict(cfg=c, sink=G.dev(csa_synth.sinks(c)), window=G.dev(win), window_host=f64(win)))
    layer = oracle_layer(cfg)
    ca, ci = oracle_comp(run.ca_host), oracle_comp(run.ci_host)
    sink_o, invf = f64(csa_synth.sinks(cfg)), f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    st_o = {b: _oracle_seq_state(host, b) for b in seqs}
    win_o = [{b: c["window_host"][b:b + 1].copy() for b in seqs} for c in cons]
    B = cfg.B
    for step in range(steps):
        si = csa_synth.step_inputs(cfg, step)
        # owner: both compress calls, its indexer and its attention (positions advance after the consumers)
        run.projs = run.compress(st, si.x)
        sel = torch.empty(B, cfg.topk, dtype=torch.int32, device="cuda")
        n_sel = torch.empty(B, dtype=torch.int32, device="cuda")
        csa.index_topk(run.L, G.dev(si.iq), G.dev(si.iw), st.ikeys, st.n_rows, st.pos, run.inv_freq, sel, n_sel,
                       err=run.err)
        out = torch.empty(B, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
        csa.attend_decode(run.L, G.dev(si.q), G.dev(si.kv), run.sink, st.window, st.pool, st.n_rows, sel, n_sel,
                          st.pos, run.inv_freq, out, err=run.err)
        torch.cuda.synchronize()
        snap = (st.pool.clone(), st.ikeys.clone(), st.n_rows.clone())
        # consumers: the index-source layer selects with its own queries; the plain one reuses the owner's selection
        c_out, c_sel = [], []
        for k, c in enumerate(cons):
            ci_in = csa_synth.step_inputs(c["cfg"], step)
            if k == 0:
                s_c = torch.empty(B, cfg.topk, dtype=torch.int32, device="cuda")
                n_c = torch.empty(B, dtype=torch.int32, device="cuda")
                csa.index_topk(run.L, G.dev(ci_in.iq), G.dev(ci_in.iw), st.ikeys, st.n_rows, st.pos, run.inv_freq,
                               s_c, n_c, err=run.err)
            else:
                s_c, n_c = sel, n_sel
            o_c = torch.empty(B, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
            csa.attend_decode(run.L, G.dev(ci_in.q), G.dev(ci_in.kv), c["sink"], c["window"], st.pool, st.n_rows,
                              s_c, n_c, st.pos, run.inv_freq, o_c, err=run.err)
            c_out.append((ci_in, o_c, s_c, n_c))
        torch.cuda.synchronize()
        assert torch.equal(st.pool, snap[0]) and torch.equal(st.ikeys, snap[1]) and torch.equal(st.n_rows, snap[2])
        st.pos += 1
        for b in seqs:
            _oracle_decode_check(layer, ca, ci, st_o[b], _step_rows(si, b), sink_o, invf, out[b].cpu(),
                                 sel[b].cpu().numpy(), n_sel[b].item(), f"owner seq {b} step {step}",
                                 _seq_projs(run, b), label="V4.1 owner layer")
            owner = dict(pool=st_o[b]["pool"], ikeys=st_o[b]["ikeys"], n_rows=st_o[b]["n_rows"],
                         pos=st_o[b]["pos"] - 1)
            p = int(owner["pos"][0])
            for k, (ci_in, o_c, s_c, n_c) in enumerate(c_out):
                xs = _step_rows(ci_in, b)
                g_sel = s_c[b].cpu().numpy()[None].astype(np.int64)
                g_n = np.array([n_c[b].item()])
                if k == 0:  # the index-source layer's own selection over the owner's keys: the gap rule
                    nv = O.visible_rows(layer, int(owner["n_rows"][0]), p)
                    scores = O.index_scores(layer, xs[3][0], xs[4][0], owner["ikeys"][0, :nv], p, invf)
                    G.check_topk(g_sel[0, :g_n[0]], scores, layer.topk, nv, what=f"consumer seq {b} top-k")
                sink_c = f64(cons[k]["sink"].cpu())
                ref, _, _, win_o[k][b], err = O.consumer_decode_step(layer, owner, win_o[k][b], xs, sink_c, invf,
                                                                     (g_sel, g_n))
                assert err == 0
                G.check_rows(o_c[b].cpu(), ref[0], "bf16", what=f"consumer {k} seq {b} step {step}", R=cfg.R,
                             label="V4.1 consumer layers")
    assert run.err.item() == 0
