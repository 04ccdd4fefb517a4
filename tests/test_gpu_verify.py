"""Verify blocks (csa_index_topk_verify, csa_attend_verify) on the GPU against the oracle.

A speculative step verifies T = K+1 tokens per sequence at once ("DeepSeek-V4-Flash: native deepseek_v4 AR backend",
MTPLX #216, "Benchmark notes"): the compressors take the block, then every query of the block gets its own causal
top-k and attention, with the prefill chunk's per-query semantics.  Checked per query against the oracle (selection
under the gap rule, output rounded and un-rounded) on a ragged batch whose first sequence crosses the dense->sparse
threshold inside a block, for several consecutive blocks; then a rejected tail is trimmed and decoding resumes.
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
    from tests.test_gpu_parity import _oracle_seq_state
    from tests.test_gpu_trim import _ragged


def _block(cfg, B, T, k):
    c = cfg.replace(cid=cfg.cid + 800)
    si = [csa_synth.step_inputs(c, 10 * k + i, B=B) for i in range(T)]
    cat = lambda f, d: torch.stack([getattr(s, f) for s in si], dim=d)  # noqa: E731
    return dict(x=torch.cat([s.x for s in si], dim=1), q=cat("q", 1), kv=cat("kv", 1), iq=cat("iq", 1), iw=cat("iw", 1))


# (B, T, compress call, sequences checked against the oracle).  B 4, T 4: the paired compress's block path, the
# indexer's 4-query MMA, the split decode attention kernel; T 5: one compress call per pool (chunk path) and the
# 1-query MMA; B 40: 160 queries, which the pipelined attention kernel takes (one CTA per query, no partials);
# T 8: two 4-query groups per sequence; B 2, T 16: 32 queries in 4 splits each, merged in-cluster.
CASES = {
    "b4_t4_pair": (4, 4, "pair", None),
    "b4_t5_per_pool": (4, 5, "single", None),
    "b40_t4_pair": (40, 4, "pair", (0, 7, 19, 33, 39)),
    "b8_t8_pair": (8, 8, "pair", (0, 5)),      # two 4-query groups per sequence; pipelined attention
    "b2_t16_pair": (2, 16, "pair", None),      # the longest block the paired compress fuses; split attention
}


@pytest.mark.parametrize("case", list(CASES))
def test_verify_blocks_against_oracle_then_trim(case):
    import deepseek_v4_compressed_csa_gb300 as csa
    B, T, mode, sampled = CASES[case]
    cfg = csa_synth.CONFIGS[3].replace(B=B, rollback=T - 1 + 8)
    if B == 4:
        ctxs = [2045, 4097, 9001, 12002]  # 2045: n_vis goes 511 -> 513 within the second block
        cap = max(ctxs) // 4 + 16
        host = _ragged(cfg, cap, ctxs)
    else:
        cfg = cfg.replace(ctx=9001)
        ctxs = [cfg.ctx] * B
        cap = cfg.ctx // 4 + 16
        host = csa_synth.synth_cache(cfg, cap)
    run = G.Runner(cfg)
    st = G.DevCache(host)
    hw = st.pos.clone()
    layer = oracle_layer(cfg)
    ca, ci = oracle_comp(run.ca_host), oracle_comp(run.ci_host)
    sink, invf = f64(csa_synth.sinks(cfg)), f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    seqs = range(cfg.B) if sampled is None else sampled
    st_o = {b: _oracle_seq_state(host, b) for b in seqs}
    label = f"verify blocks (B {B}, T {T})"
    for k in range(3):
        blk = _block(cfg, B, T, k)
        run.projs = run.compress_pair(st, blk["x"]) if mode == "pair" else run.compress(st, blk["x"])
        sel = torch.empty(B, T, cfg.topk, dtype=torch.int32, device="cuda")
        n_sel = torch.empty(B, T, dtype=torch.int32, device="cuda")
        csa.index_topk_verify(run.L, G.dev(blk["iq"]), G.dev(blk["iw"]), st.ikeys, st.n_rows, st.pos, run.inv_freq,
                              sel, n_sel, err=run.err)
        out = torch.empty(B, T, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
        csa.attend_verify(run.L, G.dev(blk["q"]), G.dev(blk["kv"]), run.sink, st.window, st.pool, st.n_rows, sel,
                          n_sel, st.pos, run.inv_freq, out, err=run.err)
        torch.cuda.synchronize()
        assert run.err.item() == 0
        g_sel, g_nsel, g_out = sel.cpu().numpy(), n_sel.cpu().numpy(), out.cpu()
        for b in seqs:
            o = st_o[b]
            p0 = int(o["pos"][0])
            x = f64(blk["x"][b:b + 1])
            n0 = o["n_rows"].copy()
            pr = {kk: v[b:b + 1].cpu() for kk, v in run.projs.items()}
            o["front_a"], o["pool"], n_a, e1 = G.oracle_compress_checked(layer, ca, x, o["pos"], o["front_a"], o["pool"],
                                                                         n0, invf, pr["attn"], f"block {k} seq {b}")
            o["front_i"], o["ikeys"], _, e2 = G.oracle_compress_checked(layer, ci, x, o["pos"], o["front_i"],
                                                                        o["ikeys"], n0, invf, pr["index"],
                                                                        f"block {k} seq {b} index")
            assert e1 == 0 and e2 == 0
            for nm, gp, op in (("pool", st.pool, o["pool"]), ("index keys", st.ikeys, o["ikeys"])):
                G.check_pool_rows(gp[b, int(n0[0]):int(n_a[0])].cpu(), op[0, int(n0[0]):int(n_a[0])], "bf16",
                                  f"block {k} seq {b} {nm}", R=cfg.R)
            o["n_rows"] = n_a
            n = int(n_a[0])
            Wr = o["window"].shape[1]
            kvr = [O.store(O.rope(f64(blk["kv"][b, i]), p0 + i, invf), "bf16") for i in range(T)]
            for i in range(T):  # the block's tokens enter the ring first
                o["window"][0, (p0 + i) % Wr] = kvr[i]
            for i in range(T):
                p = p0 + i
                nv = O.visible_rows(layer, n, p)
                rows = g_sel[b, i, :g_nsel[b, i]]
                scores = O.index_scores(layer, f64(blk["iq"][b, i]), f64(blk["iw"][b, i]), o["ikeys"][0, :nv], p,
                                        invf) if nv > layer.topk else None
                G.check_topk(rows, scores, layer.topk, nv, what=f"block {k} seq {b} query {i} top-k")
                win = [o["window"][0, t % Wr] for t in O.window_tokens(layer, p)]
                keys = np.concatenate([o["pool"][0][np.sort(rows)], np.stack(win)])
                qr = O.store(O.rope(f64(blk["q"][b, i]), p, invf), "bf16")
                att = O.attend(layer, qr, keys, sink)
                G.check_rows(g_out[b, i], O.output_rows(layer, att, p, invf), "bf16",
                             what=f"block {k} seq {b} query {i}", R=cfg.R, exact=G.exact_output(att, p, invf),
                             label=label)
            o["pos"] = o["pos"] + T
            slots = [t % Wr for t in range(p0 + T - cfg.W, p0 + T)]  # the window the next query attends
            G.check_pool_rows(st.window[b, slots].cpu(), o["window"][0, slots], "bf16", f"block {k} seq {b} ring",
                              R=cfg.R)
        csa.advance_positions(st.pos, T)
    # a speculative step keeps the first two tokens of the last block: trim the others and decode on
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_i = st.n_rows.clone()
    csa.trim(run.L, torch.full((B,), T - 2, dtype=torch.int32, device="cuda"), st.pos, st.n_rows, n_i, hw, err=err)
    si = csa_synth.step_inputs(cfg, 99, B=B)
    run.decode_step(st, si)
    torch.cuda.synchronize()
    assert err.item() == 0 and run.err.item() == 0
    assert st.pos.tolist() == [c + 2 * T + 2 + 1 for c in ctxs]


def test_verify_requires_rollback_for_the_block():
    """A block longer than the rollback margin plus one is refused on the host (its later tokens would overwrite
    window rows its earlier queries attend)."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=2, rollback=2)
    run = G.Runner(cfg)
    st = G.DevCache(_ragged(cfg, 1100, [4000, 4000]))
    z = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device="cuda")  # noqa: E731
    T = 4
    with pytest.raises(csa.CSAError) as ei:
        csa.attend_verify(run.L, z(2, T, 64, 512), z(2, T, 512), run.sink, st.window, st.pool, st.n_rows,
                          z(2, T, 512, dt=torch.int32), z(2, T, dt=torch.int32), st.pos, run.inv_freq,
                          z(2, T, 64, 512))
    assert ei.value.code == 1
