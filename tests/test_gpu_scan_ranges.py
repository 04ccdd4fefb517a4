"""The decode index scan when its CTAs' ranges of (query, key tile) items cross several queries.

The one-query scan splits B x ceil(cap / 128) items over the SMs; with many short pools a CTA's range holds several
queries, may begin in the padding tiles of its first query (past the visible rows, where that query has nothing to
score) and may reach a third query.  The blocks of a range's first two queries are prepared before the key stream
(bf16: roped by a kernel of their own and copied by TMA; fp8: the quantised codes, copied the same way) and any
other query's block is built in the loop, so these shapes reach every branch of the query-block preparation.
Checked: every sequence's selection under the gap rule against the oracle (bf16: the bf16 scores; fp8: the fp8
scores on the GPU's own query codes and key codes).
"""
import dataclasses

import numpy as np
import pytest
import torch

import csa_synth
from oracle import csa_oracle as O
from tests._common import f64, oracle_layer

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests import _gpu as G


@pytest.mark.parametrize("fp8", [False, True])
def test_scan_ranges_across_several_queries(fp8):
    import deepseek_v4_compressed_csa_gb300 as csa
    # 200 sequences of 2200 tokens (550 rows, sparse), pools of 700 rows: 6 tiles a query, the last ones padding;
    # 1200 items over the SMs, so ranges of ~8 items cross two or three queries
    cfg = csa_synth.CONFIGS[3].replace(B=200, ctx=2200)
    cap = 700
    host = csa_synth.synth_cache(cfg, cap)
    layer = oracle_layer(cfg)
    L = G.lib_layer(cfg)
    invf = f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    si = csa_synth.step_inputs(cfg.replace(cid=cfg.cid + 990), 0)
    ikeys = G.dev(host.ikeys)
    if fp8:
        L = dataclasses.replace(L, index_fp8=True)
        rows = torch.zeros(cfg.B, cap, csa.FP8_ROW_BYTES, dtype=torch.uint8, device="cuda")
        csa.index_rows_fp8(L, ikeys, rows)
        ikeys = rows
    sel = torch.empty(cfg.B, cfg.topk, dtype=torch.int32, device="cuda")
    n_sel = torch.empty(cfg.B, dtype=torch.int32, device="cuda")
    ws = torch.zeros(csa.workspace_size(L, csa.OP_INDEX_TOPK, cfg.B, 1, cap), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa.index_topk(L, G.dev(si.iq), G.dev(si.iw), ikeys, G.dev(host.n_rows), G.dev(host.pos),
                   G.dev(csa_synth.inv_freq(cfg)), sel, n_sel, ws=ws, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    g_sel, g_n = sel.cpu().numpy(), n_sel.cpu().numpy()
    p = cfg.ctx
    nv = O.visible_rows(layer, cfg.ctx // 4, p)
    assert nv > cfg.topk
    if fp8:
        a = ws.cpu().numpy()
        qc = a[:cfg.B * 8192].reshape(cfg.B, 64, 128).astype(np.int64)
        qs = np.ascontiguousarray(a[cfg.B * 8192:cfg.B * 8192 + cfg.B * 256]).view(np.float32).reshape(cfg.B, 64)
        kr = ikeys.cpu().numpy()
        kc = kr[..., :128].astype(np.int64)
        ks = np.ascontiguousarray(kr[..., 128:132]).view(np.float32)[..., 0]
    iq, iw = f64(si.iq), f64(si.iw)
    keys = f64(host.ikeys)
    for b in range(cfg.B):
        if fp8:
            scores = O.index_scores_fp8(layer, qc[b], qs[b], iw[b], kc[b, :nv], ks[b, :nv])
        else:
            scores = O.index_scores(layer, iq[b], iw[b], keys[b, :nv], p, invf)
        G.check_topk(g_sel[b][:g_n[b]], scores, cfg.topk, nv, what=f"sequence {b} ({'fp8' if fp8 else 'bf16'})")
