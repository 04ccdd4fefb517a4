"""Exact trim (csa_trim) on the GPU.

Decoding k draft tokens, rewinding them with csa_trim and then decoding the true tokens must give, bit for bit,
what decoding only the true tokens gives: the same outputs and selections at every true step and the same state
(positions, row counts, pool rows, the window tokens the next query attends, the frontier entries the next emission
pools).  The pages' rollback tests gate exactly this across a ratio-4 emission boundary, the ratio-128 boundary and
the indexer's dense-to-sparse threshold ("DeepSeek-V4-Flash: native deepseek_v4 AR backend", MTPLX #216, the MTP
post's Tests paragraph); a trim past the margin must refuse rather than rewind half-way.
"""
import pytest
import torch

import csa_synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests import _gpu as G


def _ragged(cfg, cap, ctxs):
    """One cache per sequence context (built without rollback slots, then moved into rings with them)."""
    base = cfg.replace(rollback=0)
    parts = []
    for b, c in enumerate(ctxs):
        one = csa_synth.synth_cache(base, cap, B=1, ctx=c)
        src = csa_synth.synth_cache(base, cap, B=len(ctxs), ctx=c)  # sequence b's own random stream
        for k in ("pool", "ikeys", "window", "front_attn", "front_index"):
            if getattr(one, k) is not None:
                getattr(one, k).copy_(getattr(src, k)[b:b + 1])
        n = c // cfg.ratio
        one.pool[:, n:] = 0
        if one.ikeys is not None:
            one.ikeys[:, n:] = 0
        parts.append(csa_synth.with_rollback_slots(one, cfg, c) if cfg.rollback else one)
    cat = lambda k: None if getattr(parts[0], k) is None else torch.cat([getattr(p, k) for p in parts])  # noqa: E731
    return csa_synth.Cache(**{k: cat(k) for k in vars(parts[0])})


def _decode(run, st, si):
    out, sel, n_sel = run.decode_step(st, si)
    return out.clone(), (None if sel is None else sel.clone()), (None if n_sel is None else n_sel.clone())


def _draft(cfg, B, i, j):
    return csa_synth.step_inputs(cfg.replace(cid=cfg.cid + 500), 100 * i + j, B=B)  # a stream no true step uses


def _trim(run, st, hw, k, err):
    import deepseek_v4_compressed_csa_gb300 as csa
    B = st.pos.numel()
    n_back = torch.full((B,), k, dtype=torch.int32, device="cuda") if isinstance(k, int) else k
    n_i = st.n_rows.clone() if run.cfg.has_indexer else None
    csa.trim(run.L, n_back, st.pos, st.n_rows, n_i, hw, err=err)
    if n_i is not None:
        assert torch.equal(n_i, st.n_rows)


@pytest.mark.parametrize("case", ["ratio4", "ratio128"])
def test_trim_then_redecode_is_bit_identical(case):
    if case == "ratio4":
        # 2046: the dense->sparse threshold (2051) falls inside the first drafts; all cross ratio-4 emissions
        cfg = csa_synth.CONFIGS[3].replace(B=4, rollback=64)
        ctxs, steps, drafts = [2046, 4097, 9001, 16383], 16, {2: 5, 6: 9, 11: 64}
    else:
        # 262141: the first drafts complete row 2047 (position 262143), which the true tokens then emit again
        cfg = csa_synth.CONFIGS[4].replace(B=2, rollback=32)
        ctxs, steps, drafts = [262141, 262100], 8, {0: 8, 4: 32}
    cap = max(ctxs) // cfg.ratio + (steps + 80) // cfg.ratio + 4
    host = _ragged(cfg, cap, ctxs)
    B = len(ctxs)
    run_a, run_b = G.Runner(cfg), G.Runner(cfg)
    st_a, st_b = G.DevCache(host), G.DevCache(host)
    hw = st_b.pos.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(steps):
        si = csa_synth.step_inputs(cfg, i, B=B)
        if i in drafts:
            for j in range(drafts[i]):
                _decode(run_b, st_b, _draft(cfg, B, i, j))
            _trim(run_b, st_b, hw, drafts[i], err)
        oa, sa, na = _decode(run_a, st_a, si)
        ob, sb, nb = _decode(run_b, st_b, si)
        torch.cuda.synchronize()
        assert err.item() == 0, f"step {i}: error word {err.item()}"
        assert torch.equal(oa, ob), f"step {i}: outputs differ"
        if sa is not None:
            assert torch.equal(na, nb) and torch.equal(sa, sb), f"step {i}: selections differ"
    assert run_a.err.item() == 0 and run_b.err.item() == 0
    assert torch.equal(st_a.pos, st_b.pos) and torch.equal(st_a.n_rows, st_b.n_rows)
    W, Wr, F = cfg.W, cfg.ring_slots, cfg.frontier_slots
    F0 = F - cfg.rollback
    for b in range(B):
        n, p = st_a.n_rows[b].item(), st_a.pos[b].item()
        assert torch.equal(st_a.pool[b, :n], st_b.pool[b, :n])
        if cfg.has_indexer:
            assert torch.equal(st_a.ikeys[b, :n], st_b.ikeys[b, :n])
        slots = torch.tensor([t % Wr for t in range(p - W, p)], device="cuda")
        assert torch.equal(st_a.window[b, slots], st_b.window[b, slots])
        fs = torch.tensor([t % F for t in range(p - F0, p)], device="cuda")
        assert torch.equal(st_a.front_attn[b, fs], st_b.front_attn[b, fs])
        if cfg.has_indexer:
            assert torch.equal(st_a.front_index[b, fs], st_b.front_index[b, fs])


def test_rollback_slots_change_no_result():
    """The same true tokens through rings with and without rollback slots give bit-identical outputs: the kernels
    index every ring modulo its own length and attend only the last W tokens."""
    cfg = csa_synth.CONFIGS[3].replace(B=3, rollback=48)
    ctxs = [2049, 5000, 12345]
    cap = max(ctxs) // 4 + 16
    runs = []
    for c in (cfg, cfg.replace(rollback=0)):
        run = G.Runner(c)
        st = G.DevCache(_ragged(c, cap, ctxs))
        outs = []
        for i in range(10):
            outs.append(_decode(run, st, csa_synth.step_inputs(cfg, i, B=3)))
        torch.cuda.synchronize()
        assert run.err.item() == 0
        runs.append(outs)
    for i, (x, y) in enumerate(zip(*runs)):
        assert torch.equal(x[0], y[0]) and torch.equal(x[1], y[1]), f"step {i}"


def test_trim_refuses_beyond_the_margin_and_leaves_state():
    """Per sequence: a trim past the rollback margin (counted from the highest position reached), below zero, or by
    a negative count raises CSA_DEV_ROLLBACK and leaves that sequence unchanged; the other sequences are trimmed."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=4, rollback=16)
    ctxs = [3000, 3001, 10, 4003]
    cap = max(ctxs) // 4 + 32
    run = G.Runner(cfg)
    st = G.DevCache(_ragged(cfg, cap, ctxs))
    hw = st.pos.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for j in range(12):
        _decode(run, st, _draft(cfg, 4, 0, j))
    torch.cuda.synchronize()
    p0, n0, hw0 = st.pos.clone(), st.n_rows.clone(), hw.clone()
    n_back = torch.tensor([12, 17, 23, -1], dtype=torch.int32, device="cuda")  # ok, past margin, below 0, negative
    _trim(run, st, hw, n_back, err)
    torch.cuda.synchronize()
    assert err.item() == csa.DEV_ROLLBACK
    assert st.pos.tolist() == [p0[0].item() - 12] + p0[1:].tolist()
    assert st.n_rows.tolist() == [(p0[0].item() - 12) // 4] + n0[1:].tolist()
    assert hw.tolist() == [p0[0].item()] + hw0[1:].tolist()
    # after re-decoding 6 tokens, the margin still counts from the high-water mark
    for j in range(6):
        _decode(run, st, _draft(cfg, 4, 1, j))
    err.zero_()
    _trim(run, st, hw, torch.tensor([11, 0, 0, 0], dtype=torch.int32, device="cuda"), err)
    torch.cuda.synchronize()
    assert err.item() == csa.DEV_ROLLBACK  # 3000 + 6 - 11 < 3012 - 16
    err.zero_()
    _trim(run, st, hw, torch.tensor([10, 0, 0, 0], dtype=torch.int32, device="cuda"), err)
    torch.cuda.synchronize()
    assert err.item() == 0 and st.pos[0].item() == 2996


def test_trim_into_a_prefill_chunk():
    """A prefill chunk keeps its last W + rollback window tokens and its frontier journal, so trimming 20 of its
    300 tokens and decoding on gives bit for bit what a 280-token chunk and the same decode steps give."""
    cfg = csa_synth.CONFIGS[5].replace(ctx=8192 + 2, T=300, rollback=64)
    cap = (cfg.ctx + cfg.T) // 4 + 8
    host = csa_synth.synth_cache(cfg, cap)
    ch = csa_synth.chunk_inputs(cfg)
    short = csa_synth.StepInputs(x=ch.x[:, :280], q=ch.q[:280], kv=ch.kv[:280], iq=ch.iq[:280], iw=ch.iw[:280])
    run_a, run_b = G.Runner(cfg), G.Runner(cfg)
    st_a, st_b = G.DevCache(host), G.DevCache(host)
    hw = st_b.pos.clone()
    run_a.prefill(st_a, short, cfg.ctx)
    run_b.prefill(st_b, ch, cfg.ctx)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _trim(run_b, st_b, hw, 20, err)
    torch.cuda.synchronize()
    assert err.item() == 0 and st_b.pos.item() == st_a.pos.item() == cfg.ctx + 280
    assert torch.equal(st_a.n_rows, st_b.n_rows)
    for i in range(12):  # across three ratio-4 emissions
        si = csa_synth.step_inputs(cfg, 700 + i, B=1)
        oa, sa, na = _decode(run_a, st_a, si)
        ob, sb, nb = _decode(run_b, st_b, si)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob) and torch.equal(sa, sb), f"step {i}"
    n = st_a.n_rows.item()
    assert torch.equal(st_a.pool[:, :n], st_b.pool[:, :n]) and torch.equal(st_a.ikeys[:, :n], st_b.ikeys[:, :n])
    assert run_a.err.item() == 0 and run_b.err.item() == 0
