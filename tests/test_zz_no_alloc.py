"""csa_index_topk_static: the decode indexer for callers that cannot allocate device memory.

Its scratch is a fixed array inside the library instead of a caller workspace.  It must select
exactly the rows csa_index_topk selects (the same integer result), call after call, although the
array keeps the previous call's contents, and it must not take device memory: the device's free
memory (as the driver reports it, so an allocation by the library itself would show, not only one
through torch's allocator) is the same before and after a call.  The first call on a device may
load the library's module that holds the array (the driver loads modules lazily), so the strict
check is on the second call.  This file is named to be collected last.
"""
import pytest
import torch

import csa_synth

pytestmark = pytest.mark.gpu


def _setup(B, step_seed):
    from tests import _gpu as G
    cfg = csa_synth.CONFIGS[3].replace(B=B)
    cap = cfg.ctx // cfg.ratio + 16
    host = csa_synth.synth_cache(cfg, cap, B=B)
    st = G.DevCache(host)
    si = csa_synth.step_inputs(cfg, step_seed, B=B)
    return cfg, G.lib_layer(cfg), st, G.dev(si.iq), G.dev(si.iw), G.dev(csa_synth.inv_freq(cfg))


def test_static_scratch_index_matches_workspace_version():
    import deepseek_v4_compressed_csa_gb300 as csa
    B = 8
    cfg, L, st, iq, iw, invf = _setup(B, 0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    results = []
    for call, seed in enumerate((0, 1)):  # two calls in a row, different queries
        if call:
            _, _, _, iq, iw, _ = _setup(B, seed)
        sel_ref = torch.empty(B, cfg.topk, dtype=torch.int32, device="cuda")
        nsel_ref = torch.empty(B, dtype=torch.int32, device="cuda")
        csa.index_topk(L, iq, iw, st.ikeys, st.n_rows, st.pos, invf, sel_ref, nsel_ref, err=err)
        sel = torch.full((B, cfg.topk), -7, dtype=torch.int32, device="cuda")
        nsel = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        free_before = torch.cuda.mem_get_info()[0]
        csa.index_topk_static(L, iq, iw, st.ikeys, st.n_rows, st.pos, invf, sel, nsel, err=err)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert torch.cuda.memory_allocated() == before
        if call == 0:  # at most the array itself, if this call made the driver load its module
            assert free_before - free_after <= csa.static_scratch_bytes() + (4 << 20)
        else:
            assert free_after == free_before, f"device free memory fell by {free_before - free_after} bytes"
        assert err.item() == 0
        assert torch.equal(nsel, nsel_ref) and (nsel == cfg.topk).all()  # sparse regime: 8192 rows visible
        assert torch.equal(sel, sel_ref)
        results.append(sel.clone())
    assert not torch.equal(results[0], results[1])  # the second call did not reuse the first's answer


def test_static_scratch_rejects_oversized_calls():
    """A batch whose scratch exceeds the fixed array is refused on the host, before any launch."""
    import deepseek_v4_compressed_csa_gb300 as csa
    from deepseek_v4_compressed_csa_gb300 import _binding as Bd
    cfg = csa_synth.CONFIGS[3]
    L = csa.Layer(dtype=cfg.storage, H=cfg.H, D=cfg.D, R=cfg.R, W=cfg.W, ratio=cfg.ratio, Hi=cfg.Hi, Di=cfg.Di,
                  topk=cfg.topk, X=cfg.X)
    B, cap = 256, 16
    assert csa.workspace_size(L, csa.OP_INDEX_TOPK, B, 1, cap) > csa.static_scratch_bytes()
    z = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device="cuda")  # noqa: E731
    with pytest.raises(csa.CSAError) as ei:
        csa.index_topk_static(L, z(B, 64, 128), z(B, 64), z(B, cap, 128), z(B, dt=torch.int32),
                              z(B, dt=torch.int32), z(32, dt=torch.float32), z(B, cfg.topk, dt=torch.int32),
                              z(B, dt=torch.int32))
    assert ei.value.code == Bd.CSA_ERR_WORKSPACE
