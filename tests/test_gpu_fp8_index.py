"""Index keys as fp8 rows (csa_layer.index_fp8 = 1) on the GPU against the oracle.

The mlx-lm DeepSeek-V4 port's indexer discussion (mlx-lm#1189) rotates the index operands by a Hadamard matrix and
simulates low-precision activations; this library stores the index pool as E4M3 rows of the rotated keys with one
fp32 scale per row and quantises the decode query's heads the same way (the oracle's quantize_fp8_row /
quantize_fp8_query / index_scores_fp8).  Checked here:

  * every fp8 row the compressors write (the chunk kernel and the single-token kernel of the paired call) equals,
    code for code and bit for bit in its scale, the oracle's quantisation of the row the same kernels write in the
    model dtype for a bf16 layer fed the same tokens: both sides rotate the same bf16 values with the same fp32
    butterflies, divide and round to nearest even, so nothing is left to tolerance;
  * the query codes the index call writes to its workspace: exact at position 0 (RoPE is then the identity on both
    sides, so the inputs match; an all-zero head gets scale 0 and zero codes); at later positions the GPU's fp32
    RoPE may land one bf16 ulp away from the oracle's float64 one in a few elements, so most heads must match
    exactly and every head's scale within 2^-6;
  * the selection under the gap rule against index_scores_fp8 on the GPU's own key and query codes (identical
    operands; only the summation order differs), dense (n_vis <= topk) and sparse, at every decode step; the
    fixed-scratch entry point selects the same rows.
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

ROW = 144  # bytes of an fp8 index row: 128 codes, the fp32 scale, padding


def _codes_scales(rows8: torch.Tensor):
    """uint8 [..., 144] -> (codes int64 [..., 128], scales float32 [...]); checks the zero padding."""
    a = rows8.cpu().numpy()
    assert np.all(a[..., 132:] == 0), "padding bytes of an fp8 row are not zero"
    codes = a[..., :128].astype(np.int64)
    scales = np.ascontiguousarray(a[..., 128:132]).view(np.float32)[..., 0]
    return codes, scales


def _check_rows_exact(rows8, rows16, what):
    """fp8 rows against the oracle's quantisation of the bf16 rows the same kernels wrote."""
    codes, scales = _codes_scales(rows8)
    ref = f64(rows16).astype(np.float32)
    for j in range(ref.shape[0]):
        c, s = O.quantize_fp8_row(ref[j])
        assert np.float32(s).view(np.uint32) == scales[j].view(np.uint32), f"{what} row {j}: scale {scales[j]} vs {s}"
        bad = np.nonzero(codes[j] != c)[0]
        assert bad.size == 0, f"{what} row {j}: {bad.size} codes differ, first at {bad[0]}: {codes[j, bad[0]]:#x} " \
                              f"vs {c[bad[0]]:#x}"


class _State:
    """Attention pool and index pool state of one layer on the device, from an empty cache."""

    def __init__(self, cfg, cap, fp8):
        c = csa_synth.empty_cache(cfg, cap)
        self.pool, self.front_a, self.front_i = G.dev(c.pool), G.dev(c.front_attn), G.dev(c.front_index)
        self.ikeys = (torch.zeros(cfg.B, cap, ROW, dtype=torch.uint8, device="cuda") if fp8 else G.dev(c.ikeys))
        self.n_a, self.n_i, self.pos = G.dev(c.n_rows), G.dev(c.n_rows), G.dev(c.pos)


def _query_ws(L, B, cap):
    import deepseek_v4_compressed_csa_gb300 as csa
    return torch.zeros(csa.workspace_size(L, csa.OP_INDEX_TOPK, B, 1, cap), dtype=torch.uint8, device="cuda")


def _ws_queries(ws, B):
    """The quantised decode queries in the index call's workspace: [B, 64, 128] codes, then [B, 64] fp32 scales."""
    a = ws.cpu().numpy()
    codes = a[:B * 64 * 128].reshape(B, 64, 128).astype(np.int64)
    scales = np.ascontiguousarray(a[B * 64 * 128:B * 64 * 128 + B * 64 * 4]).view(np.float32).reshape(B, 64)
    return codes, scales


def test_fp8_queries_exact_at_position_zero():
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=3, ctx=0)
    L = dataclasses.replace(G.lib_layer(cfg), index_fp8=True)
    layer = oracle_layer(cfg)
    invf = f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    cap = 64
    si = csa_synth.step_inputs(cfg.replace(cid=cfg.cid + 900), 0)
    iq = si.iq.clone()
    iq[1, 5] = 0  # an all-zero head: scale 0, zero codes
    st = _State(cfg, cap, True)
    sel = torch.empty(cfg.B, cfg.topk, dtype=torch.int32, device="cuda")
    n_sel = torch.empty(cfg.B, dtype=torch.int32, device="cuda")
    ws = _query_ws(L, cfg.B, cap)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa.index_topk(L, G.dev(iq), G.dev(si.iw), st.ikeys, st.n_i, st.pos, G.dev(csa_synth.inv_freq(cfg)), sel, n_sel,
                   ws=ws, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert n_sel.cpu().tolist() == [0] * cfg.B
    codes, scales = _ws_queries(ws, cfg.B)
    for b in range(cfg.B):
        c, s = O.quantize_fp8_query(layer, f64(iq[b]), 0, invf)
        assert np.array_equal(scales[b].view(np.uint32), s.view(np.uint32)), f"query {b}: scales differ"
        assert np.array_equal(codes[b], c), f"query {b}: codes differ"
    assert scales[1, 5] == 0 and not codes[1, 5].any()


def test_index_rows_fp8_conversion():
    """csa_index_rows_fp8 on seeded rows, with an all-zero row, rows scaled far up and down (E4M3 subnormal codes,
    bf16 subnormal inputs) and a row with one dominant element (every other code small): bit-exact."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=2, ctx=4 * 300)
    L = dataclasses.replace(G.lib_layer(cfg), index_fp8=True)
    src = csa_synth.synth_cache(cfg, 300).ikeys.clone()  # [2, 300, 128] seeded N(0,1), bf16
    src[0, 0] = 0
    src[0, 1] *= 1e30
    src[0, 2] *= 1e-38
    src[1, 3] *= 1e-3
    src[1, 3, 17] = 1e3
    dst = torch.zeros(2, 300, ROW, dtype=torch.uint8, device="cuda")
    csa.index_rows_fp8(L, G.dev(src), dst)
    torch.cuda.synchronize()
    _check_rows_exact(dst.view(-1, ROW), src.view(-1, 128), "converted")
    codes, scales = _codes_scales(dst[0, 0])
    assert scales == 0 and not codes.any()


# (tokens compressed from an empty cache before the decode steps, decode steps): 1023 tokens leave 255 rows
# (dense: every visible row is selected), 4095 leave 1023 rows (sparse: 512 of 1023 .. 1024).
CASES = {"dense": (1023, 6), "sparse": (4095, 6)}


@pytest.mark.parametrize("case", list(CASES))
def test_fp8_index_rows_and_selection(case):
    import deepseek_v4_compressed_csa_gb300 as csa
    T0, steps = CASES[case]
    cfg = csa_synth.CONFIGS[3].replace(B=2, ctx=0)
    L16 = G.lib_layer(cfg)
    L8 = dataclasses.replace(L16, index_fp8=True)
    layer = oracle_layer(cfg)
    invf = f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    inv_freq = G.dev(csa_synth.inv_freq(cfg))
    ca = G.lib_comp(csa_synth.compressor(cfg, "attn"))
    ci = G.lib_comp(csa_synth.compressor(cfg, "index"))
    cap = (T0 + steps) // 4 + 70  # ragged last tile of 128 rows
    s16, s8 = _State(cfg, cap, False), _State(cfg, cap, True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the cache: one chunk of T0 tokens per sequence through each pool's own compress call (chunk kernel)
    x = G.dev(csa_synth.hidden(cfg, T0, tag=31))
    for L, s in ((L16, s16), (L8, s8)):
        csa.compress_append(L, ca, x, s.pos, s.front_a, s.pool, s.n_a, inv_freq, err=err)
        csa.compress_append(L, ci, x, s.pos, s.front_i, s.ikeys, s.n_i, inv_freq, err=err)
        s.pos += T0
    torch.cuda.synchronize()
    assert err.item() == 0
    n0 = T0 // 4
    assert s8.n_i.cpu().tolist() == [n0] * cfg.B
    for b in range(cfg.B):
        _check_rows_exact(s8.ikeys[b, :n0], s16.ikeys[b, :n0], f"chunk, sequence {b}")
    assert torch.equal(s8.pool, s16.pool)
    conv = torch.zeros(cfg.B, n0, ROW, dtype=torch.uint8, device="cuda")
    csa.index_rows_fp8(L8, s16.ikeys[:, :n0].contiguous(), conv)
    assert torch.equal(conv, s8.ikeys[:, :n0]), "csa_index_rows_fp8 differs from the compress kernels' fp8 rows"
    mism, heads = 0, 0
    for k in range(steps):
        si = csa_synth.step_inputs(cfg.replace(cid=cfg.cid + 900), k + 1)
        xk = G.dev(si.x)
        for L, s in ((L16, s16), (L8, s8)):  # both pools in one call: the single-token kernel
            csa.compress_append_pair(L, ca, ci, xk, s.pos, s.front_a, s.pool, s.n_a, s.front_i, s.ikeys, s.n_i,
                                     inv_freq, err=err)
        sel = torch.empty(cfg.B, cfg.topk, dtype=torch.int32, device="cuda")
        n_sel = torch.empty(cfg.B, dtype=torch.int32, device="cuda")
        ws = _query_ws(L8, cfg.B, cap)
        iq, iw = G.dev(si.iq), G.dev(si.iw)
        csa.index_topk(L8, iq, iw, s8.ikeys, s8.n_i, s8.pos, inv_freq, sel, n_sel, ws=ws, err=err)
        sel_s = torch.empty_like(sel)
        n_sel_s = torch.empty_like(n_sel)
        csa.index_topk_static(L8, iq, iw, s8.ikeys, s8.n_i, s8.pos, inv_freq, sel_s, n_sel_s, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.equal(sel_s, sel) and torch.equal(n_sel_s, n_sel)
        n = s8.n_i.cpu().numpy()
        pos = s8.pos.cpu().numpy()
        assert np.array_equal(n, s16.n_i.cpu().numpy())
        if (pos[0] + 1) % 4 == 0:  # the step completed a row: the single-token kernel's fp8 store
            for b in range(cfg.B):
                _check_rows_exact(s8.ikeys[b, n[b] - 1:n[b]], s16.ikeys[b, n[b] - 1:n[b]], f"step {k}, seq {b}")
        qc, qs = _ws_queries(ws, cfg.B)
        kc, ks = _codes_scales(s8.ikeys)
        g_sel, g_n = sel.cpu().numpy(), n_sel.cpu().numpy()
        for b in range(cfg.B):
            p = int(pos[b])
            oc, osc = O.quantize_fp8_query(layer, f64(si.iq[b]), p, invf)
            rel = np.abs(qs[b].astype(np.float64) - osc) / np.maximum(osc, 1e-30)
            assert rel.max() <= 2.0 ** -6, f"step {k} seq {b}: query scale off by {rel.max()}"
            same = np.all(qc[b] == oc, axis=1)
            mism += int((~same).sum())
            heads += same.size
            nv = O.visible_rows(layer, int(n[b]), p)
            rows = g_sel[b][:g_n[b]]
            scores = O.index_scores_fp8(layer, qc[b], qs[b], f64(si.iw[b]), kc[b, :nv], ks[b, :nv])
            G.check_topk(rows, scores, layer.topk, nv, what=f"step {k} seq {b} fp8 top-k")
        s8.pos += 1
        s16.pos += 1
    # a head's codes differ only when the fp32 RoPE of one of its elements rounds to the other bf16 neighbour
    assert mism <= heads // 10, f"{mism} of {heads} query heads quantised differently from the oracle"


def _fp8_cache(cfg, T0, cap, tag):
    """Both pools of B sequences from T0 seeded tokens each, the index pool as fp8 rows (the chunk kernel)."""
    import deepseek_v4_compressed_csa_gb300 as csa
    L8 = dataclasses.replace(G.lib_layer(cfg), index_fp8=True)
    ca = G.lib_comp(csa_synth.compressor(cfg, "attn"))
    ci = G.lib_comp(csa_synth.compressor(cfg, "index"))
    s = _State(cfg, cap, True)
    s.window = G.dev(csa_synth.empty_cache(cfg, cap).window)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    inv_freq = G.dev(csa_synth.inv_freq(cfg))
    if T0:
        x = G.dev(csa_synth.hidden(cfg, T0, tag=tag))
        csa.compress_append(L8, ca, x, s.pos, s.front_a, s.pool, s.n_a, inv_freq, err=err)
        csa.compress_append(L8, ci, x, s.pos, s.front_i, s.ikeys, s.n_i, inv_freq, err=err)
        s.pos += T0
    torch.cuda.synchronize()
    assert err.item() == 0
    return L8, ca, ci, s, err, inv_freq


def _check_queries(layer, ws, off, Q, iws, ikeys_b, n_rows, positions, sel, n_sel, what):
    """Selections of Q queries (query i of sequence seq[i] at position positions[i]) against the fp8 scores on the
    GPU's own query codes (in ws at byte off) and key codes."""
    a = ws.cpu().numpy()[off:]
    qc = a[:Q * 64 * 128].reshape(Q, 64, 128).astype(np.int64)
    qs = np.ascontiguousarray(a[Q * 64 * 128:Q * 64 * 128 + Q * 256]).view(np.float32).reshape(Q, 64)
    g_sel, g_n = sel.cpu().numpy().reshape(Q, -1), n_sel.cpu().numpy().reshape(Q)
    for i in range(Q):
        kc, ks = _codes_scales(ikeys_b(i))
        nv = O.visible_rows(layer, int(n_rows(i)), int(positions[i]))
        scores = O.index_scores_fp8(layer, qc[i], qs[i], iws[i], kc[:nv], ks[:nv])
        G.check_topk(g_sel[i][:g_n[i]], scores, layer.topk, nv, what=f"{what} query {i}")


@pytest.mark.parametrize("T", [4, 5])
def test_fp8_verify_blocks(T):
    """Verify blocks on fp8 rows: T = 4 scores four queries per product (the 4-query instance), T = 5 one."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=2, ctx=0, rollback=T - 1 + 4)
    T0 = 2047
    cap = (T0 + 3 * T) // 4 + 40
    L8, ca, ci, s, err, inv_freq = _fp8_cache(cfg, T0, cap, 51)
    layer = oracle_layer(cfg)
    for k in range(2):  # the second block crosses 512 visible rows for some queries
        blk = [csa_synth.step_inputs(cfg.replace(cid=cfg.cid + 960 + k), i) for i in range(T)]
        x = G.dev(torch.cat([b.x for b in blk], dim=1))
        csa.compress_append_pair(L8, ca, ci, x, s.pos, s.front_a, s.pool, s.n_a, s.front_i, s.ikeys, s.n_i, inv_freq,
                                 err=err)
        iq = torch.stack([b.iq for b in blk], 1)
        iw = torch.stack([b.iw for b in blk], 1)
        sel = torch.empty(cfg.B, T, cfg.topk, dtype=torch.int32, device="cuda")
        n_sel = torch.empty(cfg.B, T, dtype=torch.int32, device="cuda")
        ws = torch.zeros(csa.workspace_size(L8, csa.OP_INDEX_TOPK, cfg.B * T, 1, cap), dtype=torch.uint8,
                         device="cuda")
        csa.index_topk_verify(L8, G.dev(iq), G.dev(iw), s.ikeys, s.n_i, s.pos, inv_freq, sel, n_sel, ws=ws, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        pos = s.pos.cpu().numpy()
        n = s.n_i.cpu().numpy()
        Q = cfg.B * T
        _check_queries(layer, ws, 0, Q, f64(iw).reshape(Q, -1), lambda i: s.ikeys[i // T], lambda i: n[i // T],
                       [pos[i // T] + i % T for i in range(Q)], sel, n_sel, f"verify block {k}")
        csa.advance_positions(s.pos, T)


def test_fp8_prefill_chunk_and_varlen():
    """A prefill chunk (one sequence) and a packed batch on fp8 rows, both through the 4-query instance (the packed
    batch from its group table); selections against the fp8 scores on the GPU's codes."""
    import deepseek_v4_compressed_csa_gb300 as csa
    cfg = csa_synth.CONFIGS[3].replace(B=1, ctx=0)
    T0, T = 2099, 41
    cap = (T0 + T) // 4 + 30
    L8, ca, ci, s, err, inv_freq = _fp8_cache(cfg, T0, cap, 52)
    layer = oracle_layer(cfg)
    ch = csa_synth.chunk_inputs(cfg.replace(cid=cfg.cid + 970), T)
    x = G.dev(ch.x)
    n_i = s.n_i
    csa.compress_append(L8, ca, x, s.pos, s.front_a, s.pool, s.n_a, inv_freq, err=err)
    csa.compress_append(L8, ci, x, s.pos, s.front_i, s.ikeys, n_i, inv_freq, err=err)
    out = torch.empty(T, cfg.H, cfg.D, dtype=cfg.storage, device="cuda")
    sel = torch.empty(T, cfg.topk, dtype=torch.int32, device="cuda")
    ws = torch.zeros(csa.workspace_size(L8, csa.OP_ATTEND_PREFILL, 1, T, cap), dtype=torch.uint8, device="cuda")
    csa.attend_prefill_chunk(L8, G.dev(ch.q), G.dev(ch.kv), G.dev(ch.iq), G.dev(ch.iw), G.dev(csa_synth.sinks(cfg)),
                             T0, s.window[0], s.pool[0], s.ikeys[0], s.n_a, inv_freq, out, sel_out=sel, ws=ws, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    n = int(s.n_a.item())
    n_sel = torch.tensor([int((sel[i] >= 0).sum()) for i in range(T)], dtype=torch.int32)
    _check_queries(layer, ws, 0, T, f64(ch.iw), lambda i: s.ikeys[0], lambda i: n, [T0 + i for i in range(T)], sel,
                   n_sel, "prefill")
    # a packed batch: a sequence of 2099 tokens takes 9 more, one of 2051 takes 30, one empty chunk in between
    cfgv = csa_synth.CONFIGS[3].replace(B=3, ctx=0)
    lens = [9, 0, 30]
    T0v = 2099
    capv = (T0v + 40) // 4 + 30
    L8, ca, ci, sv, err, inv_freq = _fp8_cache(cfgv, T0v, capv, 53)
    N = sum(lens)
    cu = torch.tensor([0, 9, 9, 39], dtype=torch.int32, device="cuda")
    chv = csa_synth.chunk_inputs(cfgv.replace(cid=cfgv.cid + 980), N)
    xv = G.dev(chv.x[0])
    csa.compress_append_varlen(L8, ca, xv, cu, max(lens), sv.pos, sv.front_a, sv.pool, sv.n_a, inv_freq, err=err)
    csa.compress_append_varlen(L8, ci, xv, cu, max(lens), sv.pos, sv.front_i, sv.ikeys, sv.n_i, inv_freq, err=err)
    out = torch.empty(N, cfgv.H, cfgv.D, dtype=cfgv.storage, device="cuda")
    sel = torch.empty(N, cfgv.topk, dtype=torch.int32, device="cuda")
    ws = torch.zeros(csa.workspace_size(L8, csa.OP_ATTEND_PREFILL_VARLEN, 3, N, capv), dtype=torch.uint8,
                     device="cuda")
    csa.attend_prefill_varlen(L8, G.dev(chv.q), G.dev(chv.kv), G.dev(chv.iq), G.dev(chv.iw),
                              G.dev(csa_synth.sinks(cfgv)), cu, max(lens), sv.pos, sv.window, sv.pool, sv.ikeys, sv.n_a,
                              inv_freq, out, sel_out=sel, ws=ws, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    seq = [0] * 9 + [2] * 30
    posq = [T0v + i for i in range(9)] + [T0v + i for i in range(30)]
    nv = sv.n_a.cpu().numpy()
    n_sel = torch.tensor([int((sel[i] >= 0).sum()) for i in range(N)], dtype=torch.int32)
    off = (4 * 4 + 255) // 256 * 256  # the group table of 3 + 1 entries comes first
    _check_queries(layer, ws, off, N, f64(chv.iw), lambda i: sv.ikeys[seq[i]], lambda i: nv[seq[i]], posq, sel, n_sel,
                   "varlen")
