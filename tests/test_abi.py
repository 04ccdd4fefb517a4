"""The C ABI without a GPU: the library loads, exports every function include/csa.h declares, and rejects
bad arguments on the host (synchronously, before touching the device)."""
import ctypes
import os
import re

import pytest

import deepseek_v4_compressed_csa_gb300 as csa
from deepseek_v4_compressed_csa_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from deepseek_v4_compressed_csa_gb300 import build
        build.build()
    return csa.load_library()


def _declared_functions():
    names = []
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:[A-Za-z_][A-Za-z0-9_]*[\s*]+)+(csa_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert set(declared) >= {"csa_compress_append", "csa_index_topk", "csa_attend_decode",
                             "csa_attend_prefill_chunk", "csa_workspace_size"}
    for name in declared:
        assert hasattr(lib, name), f"libcsa.so does not export {name}"
    assert set(B.EXPORTS) <= set(declared)


def _layer(**kw):
    base = dict(dtype=B.CSA_BF16, H=64, D=512, R=64, W=128, ratio=4, Hi=64, Di=128, topk=512, X=4096, scale=0.0,
                rms_eps=1e-6, rollback=0, index_fp8=0)
    base.update(kw)
    return B._Layer(*[base[f] for f, _ in B._Layer._fields_])


def test_frontier_slots_and_status_strings(lib):
    assert lib.csa_frontier_slots(4) == 8
    assert lib.csa_frontier_slots(128) == 128
    assert lib.csa_status_string(0) == b"CSA_OK"
    assert b"WORKSPACE" in lib.csa_status_string(4)


def test_workspace_sizes(lib):
    L = _layer()
    n = ctypes.c_size_t()
    sizes = {}
    for op in (B.OP_COMPRESS, B.OP_INDEX_TOPK, B.OP_ATTEND_DECODE, B.OP_ATTEND_PREFILL):
        assert lib.csa_workspace_size(ctypes.byref(L), op, 32, 4, 8400, ctypes.byref(n)) == 0
        sizes[op] = n.value
        assert n.value > 0
    assert lib.csa_workspace_size(ctypes.byref(L), B.OP_INDEX_TOPK, 64, 1, 8400, ctypes.byref(n)) == 0
    assert n.value > sizes[B.OP_INDEX_TOPK]
    assert lib.csa_workspace_size(ctypes.byref(L), 99, 1, 1, 1, ctypes.byref(n)) == B.CSA_ERR_ARG
    assert lib.csa_workspace_size(ctypes.byref(_layer(D=500)), 0, 1, 1, 1, ctypes.byref(n)) == B.CSA_ERR_ARG


FAKE = 0x7f0000000000  # never dereferenced: every call below fails validation first


def _compress(lib, L, comp=None, ws_bytes=0, x=FAKE, pos=FAKE, err=FAKE, T=4):
    comp = comp or B._Comp(FAKE, FAKE, FAKE, FAKE, 512)
    return lib.csa_compress_append(ctypes.byref(L) if L is not None else None, ctypes.byref(comp), x, 2, T, pos,
                                   FAKE, FAKE, 100, FAKE, FAKE, FAKE, ws_bytes, err, None)


def test_host_validation_fails_closed(lib):
    L = _layer()
    assert _compress(lib, None) == B.CSA_ERR_ARG
    assert _compress(lib, _layer(dtype=7)) == B.CSA_ERR_ARG
    assert _compress(lib, _layer(R=60)) == B.CSA_ERR_ARG
    assert _compress(lib, _layer(X=4100)) == B.CSA_ERR_ARG
    assert _compress(lib, L, comp=B._Comp(FAKE, FAKE, FAKE, FAKE, 100)) == B.CSA_ERR_ARG
    assert _compress(lib, L, x=FAKE + 2) == B.CSA_ERR_ARG
    assert _compress(lib, L, x=0) == B.CSA_ERR_ARG
    assert _compress(lib, L, pos=FAKE + 2) == B.CSA_ERR_ARG
    assert _compress(lib, L, T=0) == B.CSA_ERR_ARG
    assert _compress(lib, L, ws_bytes=16) == B.CSA_ERR_WORKSPACE
    # the index call exists only for layers with an indexer
    L128 = _layer(ratio=128)
    assert lib.csa_index_topk(ctypes.byref(L128), FAKE, FAKE, 1, FAKE, 10, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                              1 << 30, FAKE, None) == B.CSA_ERR_UNSUPPORTED
    # decode attention: selections on a layer without an indexer are rejected
    assert lib.csa_attend_decode(ctypes.byref(L128), FAKE, FAKE, FAKE, 1, FAKE, FAKE, 10, FAKE, FAKE, FAKE, FAKE,
                                 FAKE, FAKE, FAKE, 1 << 30, FAKE, None) == B.CSA_ERR_ARG
    # trim: a negative rollback capacity, null state pointers, a layer with an indexer without its n_rows
    assert lib.csa_trim(ctypes.byref(_layer(rollback=-1)), 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == B.CSA_ERR_ARG
    assert lib.csa_trim(ctypes.byref(L), 2, FAKE, None, FAKE, FAKE, FAKE, FAKE, None) == B.CSA_ERR_ARG
    assert lib.csa_trim(ctypes.byref(L), 2, FAKE, FAKE, FAKE, None, FAKE, FAKE, None) == B.CSA_ERR_ARG
    assert lib.csa_trim(ctypes.byref(L), 0, None, None, None, None, None, None, None) == B.CSA_OK
    # prefill: chunk length bounds and a too-small workspace
    args = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert lib.csa_attend_prefill_chunk(ctypes.byref(L), *args, 0, 0, FAKE, FAKE, FAKE, 10, FAKE, FAKE, FAKE, None,
                                        FAKE, 1 << 30, FAKE, None) == B.CSA_ERR_ARG
    assert lib.csa_attend_prefill_chunk(ctypes.byref(L), *args, 8, 0, FAKE, FAKE, FAKE, 10, FAKE, FAKE, FAKE, None,
                                        FAKE, 64, FAKE, None) == B.CSA_ERR_WORKSPACE


def test_binding_requires_cuda_tensors(lib):
    import torch
    L = csa.Layer(dtype=torch.bfloat16, H=64, D=512, R=64, W=128, ratio=4, Hi=64, Di=128, topk=512, X=4096)
    with pytest.raises(ValueError):
        B._ptr(torch.zeros(4))
    assert csa.workspace_size(L, csa.OP_ATTEND_DECODE, 32, 1, 8400) > 0


def _decode_args(torch, dt=None, **over):
    """Arguments of attend_decode for B = 2 with the right dtypes and shapes (CPU tensors: nothing here may
    reach the device), with ``over`` replacing some of them."""
    dt = dt or torch.bfloat16
    B_, H, D, W, cap, k = 2, 64, 512, 128, 40, 512
    a = dict(q=torch.zeros(B_, H, D, dtype=dt), kv_new=torch.zeros(B_, D, dtype=dt),
             sink=torch.zeros(H, dtype=torch.float32), window=torch.zeros(B_, W, D, dtype=dt),
             pool=torch.zeros(B_, cap, D, dtype=dt), n_rows=torch.zeros(B_, dtype=torch.int32),
             sel=torch.zeros(B_, k, dtype=torch.int32), n_sel=torch.zeros(B_, dtype=torch.int32),
             pos=torch.zeros(B_, dtype=torch.int32), inv_freq=torch.zeros(32, dtype=torch.float32),
             out=torch.zeros(B_, H, D, dtype=dt))
    a.update(over)
    return a


def test_binding_checks_dtypes_and_shapes_before_the_device(lib):
    """The C ABI takes untyped pointers, so the binding checks every tensor's dtype and shape against the layer
    and the call first: a wrong dtype raises TypeError and a wrong shape ValueError before any allocation, device
    check or launch (here with CPU tensors, which would otherwise fail only at the device check)."""
    import torch
    L = csa.Layer(dtype=torch.bfloat16, H=64, D=512, R=64, W=128, ratio=4, Hi=64, Di=128, topk=512, X=4096)
    with pytest.raises(ValueError, match="CUDA"):  # everything right: only the device check is left
        csa.attend_decode(L, **_decode_args(torch))
    bad_dtype = [("q", torch.zeros(2, 64, 512)), ("sink", torch.zeros(64, dtype=torch.bfloat16)),
                 ("n_rows", torch.zeros(2, dtype=torch.int64)), ("sel", torch.zeros(2, 512)),
                 ("inv_freq", torch.zeros(32, dtype=torch.float64)), ("out", torch.zeros(2, 64, 512))]
    for name, t in bad_dtype:
        with pytest.raises(TypeError, match=name):
            csa.attend_decode(L, **_decode_args(torch, **{name: t}))
    bad_shape = [("q", torch.zeros(2, 64, 256, dtype=torch.bfloat16)),
                 ("kv_new", torch.zeros(3, 512, dtype=torch.bfloat16)),
                 ("window", torch.zeros(2, 64, 512, dtype=torch.bfloat16)),
                 ("sel", torch.zeros(2, 256, dtype=torch.int32)), ("pos", torch.zeros(1, dtype=torch.int32))]
    for name, t in bad_shape:
        with pytest.raises(ValueError, match=name):
            csa.attend_decode(L, **_decode_args(torch, **{name: t}))
    # the other calls: an fp32 tensor handed to a bf16 layer
    z = torch.zeros
    with pytest.raises(TypeError, match="iq"):
        csa.index_topk(L, z(2, 64, 128), z(2, 64, dtype=torch.bfloat16), z(2, 40, 128, dtype=torch.bfloat16),
                       z(2, dtype=torch.int32), z(2, dtype=torch.int32), z(32), z(2, 512, dtype=torch.int32),
                       z(2, dtype=torch.int32))
    comp = csa.Compressor(wkv=z(1024, 4096, dtype=torch.bfloat16), wgate=z(1024, 4096, dtype=torch.bfloat16),
                          ape=z(4, 1024), norm_w=z(512), d=512)
    with pytest.raises(TypeError, match="x"):
        csa.compress_append(L, comp, z(2, 1, 4096), z(2, dtype=torch.int32), z(2, 8, 2048, dtype=torch.bfloat16),
                            z(2, 40, 512, dtype=torch.bfloat16), z(2, dtype=torch.int32), z(32))
    with pytest.raises(ValueError, match="frontier"):
        csa.compress_append(L, comp, z(2, 1, 4096, dtype=torch.bfloat16), z(2, dtype=torch.int32),
                            z(2, 4, 2048, dtype=torch.bfloat16), z(2, 40, 512, dtype=torch.bfloat16),
                            z(2, dtype=torch.int32), z(32))


def test_fp8_index_rows_host_checks(lib):
    """index_fp8: 0 or 1; fp8 rows need ratio 4, bf16, Hi = 64, Di = 128, R <= 64 and D != Di; the overlapped index
    call refuses such a layer before touching a pointer."""
    n = ctypes.c_size_t()
    assert lib.csa_workspace_size(ctypes.byref(_layer(index_fp8=1)), B.OP_INDEX_TOPK, 32, 1, 8400,
                                  ctypes.byref(n)) == B.CSA_OK
    assert lib.csa_workspace_size(ctypes.byref(_layer(index_fp8=2)), 0, 1, 1, 1, ctypes.byref(n)) == B.CSA_ERR_ARG
    for bad in (dict(ratio=128), dict(dtype=B.CSA_F32), dict(Hi=32), dict(Di=64, R=64), dict(D=128), dict(R=72)):
        assert lib.csa_workspace_size(ctypes.byref(_layer(index_fp8=1, **bad)), 0, 1, 1, 1,
                                      ctypes.byref(n)) == B.CSA_ERR_UNSUPPORTED, bad
    L8 = _layer(index_fp8=1, rollback=8)
    assert lib.csa_index_topk_overlapped(ctypes.byref(L8), FAKE, FAKE, 1, FAKE, 10, FAKE, FAKE, FAKE, FAKE, FAKE,
                                         FAKE, 1 << 30, FAKE, None, None) == B.CSA_ERR_UNSUPPORTED


def test_index_rows_fp8_host_checks(lib):
    L8, L16 = _layer(index_fp8=1), _layer()
    assert lib.csa_index_rows_fp8(ctypes.byref(L16), FAKE, 4, FAKE, None) == B.CSA_ERR_UNSUPPORTED
    assert lib.csa_index_rows_fp8(ctypes.byref(L8), FAKE, -1, FAKE, None) == B.CSA_ERR_ARG
    assert lib.csa_index_rows_fp8(ctypes.byref(L8), FAKE + 8, 4, FAKE, None) == B.CSA_ERR_ARG
    assert lib.csa_index_rows_fp8(ctypes.byref(L8), FAKE, 4, None, None) == B.CSA_ERR_ARG
    assert lib.csa_index_rows_fp8(ctypes.byref(L8), None, 0, None, None) == B.CSA_OK  # nothing to do
